// Backward attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), for
// f16 / bf16 inputs, D in {64, 128}.
//
// The fused backward of the OCANNL "Module Ir.Online_softmax" page (third
// bullet): a per-row Dr = sum(dO * O) (the preprocess kernel), then nests that
// recompute each pair's p, dp and ds = p * (dp - Dr) -- one over the keys
// accumulating dk and dv, one over the query rows accumulating dq, each owning
// what it writes (no atomics; results are run-to-run deterministic).
//
// dkdv kernel -- work item = 128 keys of one (sequence, head); loop over the
// 128-row query blocks that can see them.  Per block, with the key tile as the
// MMA's M dimension (TMEM lane = key):
//   S^T  = K Q^T          (smem x smem)            -> TMEM [0, 128)
//   dP^T = V dO^T         (smem x smem)            -> TMEM [128, 256)
//   P^T  = 2^(S^T * scale * log2e - lse2[q])       elementwise warps, 16-bit into TMEM over S^T
//   dV  += P^T dO         (TMEM x smem, dO N-major) -> TMEM [256, 256 + D)
//   dS^T = P^T (dP^T - Dr[q])                      elementwise, 16-bit into TMEM over dP^T
//   dK  += dS^T Q         (TMEM x smem, Q N-major)  -> TMEM [256 + D, 256 + 2D)
// MMA issue order dV_i, S_{i+1}, dK_i, dP_{i+1} overlaps the elementwise work
// of one block with the contractions of the next.
//
// dq kernel -- work item = 128 query rows; loop over key blocks:
//   S = Q K^T, dP = dO V^T into TMEM, each with its own commit; the
//   elementwise warps read S into registers (freeing its buffer for the next
//   block's S), exponentiate it, then read dP (freeing that buffer), form
//   dS = P (dP - Dr) and write it, 16-bit, into one of two TMEM buffers;
//   dQ += dS K (TMEM x smem, K N-major).  Issue order S_{j+1}, dP_{j+1}, dQ_j.
//
// Warp roles (12 warps): 0 TMA producer, 1 MMA issuer (the whole warp runs
// the loop, one elected lane issues), 4-11 two elementwise warpgroups that
// split each row's 128 columns in halves.  lse2 =
// lse * log2(e) and Dr come from the preprocess kernel.  All waits bounded.
#include "sm100.cuh"
#include "tc.h"

namespace attn {

namespace {

using namespace sm100;

constexpr int BT = 128;           // rows of a query tile = keys of a key tile
constexpr int kThreads = 384;
constexpr int kEw = 256;          // elementwise threads (warps 4-11)
constexpr int kSchedConsumers = 1 + 8;

template <int D>
struct BCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = 128 * 64 * 2;
    static constexpr int kTileBytes = 128 * D * 2;
    // dkdv: Q tiles stay until dK of their block, dO tiles only until dV
    static constexpr int kDkdvQStages = D == 128 ? 2 : 4;
    static constexpr int kDkdvDoStages = D == 128 ? 2 : 4;
    // dq: K tiles stay until dQ of their block, V tiles only until its dP, so
    // the K ring is deeper; both prefetch far enough ahead to hide L2 latency
    static constexpr int kDqKStages = D == 128 ? 3 : 5;
    static constexpr int kDqVStages = D == 128 ? 2 : 3;
    // fused dQ: the 16-bit dS tile (128 keys x 128 query rows, 32 KiB) for the
    // dQ contraction lives in the dO ring slot of its block at D = 128 (same
    // size; dO is dead once dP^T is done) and in a buffer of its own at D = 64
    static constexpr int kDsBytes = BT * BT * 2;
    static constexpr bool kDsInDoSlot = kTileBytes == kDsBytes;
    static constexpr int kDkdvSmem =
        (2 + kDkdvQStages + kDkdvDoStages) * kTileBytes + (kDsInDoSlot ? 0 : kDsBytes) + 1024;
    // fused dQ accumulator columns: at D = 128 TMEM is full (S^T, dP^T, dV, dK),
    // so dQ of a block reuses the dP^T columns once its dS^T has been consumed
    static constexpr uint32_t kDqCol = D == 128 ? BT : 256 + 2 * D;
    static constexpr int kDqSmem = (2 + kDqKStages + kDqVStages) * kTileBytes + 1024;
    // dynamic + static (barriers, stats) shared memory within the 227 KiB per block
    static_assert(kDkdvSmem + 3 * 1024 <= 232448 && kDqSmem + 1024 <= 232448, "shared memory budget");
    static constexpr int kRegsProducer = 88;
    static constexpr int kRegsEw = 208;
    static_assert(128 * kRegsProducer + 256 * kRegsEw <= kThreads * 168, "register split");
    // fused dQ: the MMA issuer keeps more descriptors and counters live
    static constexpr int kRegsProducerFused = 112;
    static constexpr int kRegsEwFused = 184;
    static_assert(128 * kRegsProducerFused + 256 * kRegsEwFused <= kThreads * 168, "register split");
};

struct TcBwdArgs {
    CUtensorMap tq, tk, tv, tdo;
    BwdParams p;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

constexpr long long kDrainCycles = 1ll << 31;  // post-abort wait for TMA loads in flight

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long budget) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) return;
    }
}

// The scheduler ring shared by both kernels: the producer fetches item
// indices from the global counter, the MMA thread and 8 elementwise warps read them.
struct SchedRing {
    uint64_t full[2], empty[2];
    int item[2];
};

__device__ __forceinline__ bool sched_publish(SchedRing &r, int i, int *counter, int &w, const Watchdog &wd) {
    const int slot = i & 1;
    if (!mbar_wait(smem_u32(&r.empty[slot]), ((i >> 1) & 1) ^ 1, wd)) return false;
    w = atomicAdd(counter, 1);
    r.item[slot] = w;
    mbar_arrive(smem_u32(&r.full[slot]));
    return true;
}

__device__ __forceinline__ bool sched_take(SchedRing &r, int i, int &w, const Watchdog &wd) {
    const int slot = i & 1;
    if (!mbar_wait(smem_u32(&r.full[slot]), (i >> 1) & 1, wd)) return false;
    w = r.item[slot];
    mbar_arrive(smem_u32(&r.empty[slot]));
    return true;
}

// warp-wide versions: every lane waits (the same observations), one lane
// fetches / arrives, every lane gets the item
__device__ __forceinline__ bool sched_publish_warp(SchedRing &r, int i, int *counter, int &w, const Watchdog &wd) {
    const int slot = i & 1;
    const bool ok = mbar_wait(smem_u32(&r.empty[slot]), ((i >> 1) & 1) ^ 1, wd);
    if (!__all_sync(0xffffffffu, ok)) return false;
    int v = 0;
    const bool lead = elect_one();
    if (lead) {
        v = atomicAdd(counter, 1);
        r.item[slot] = v;
        mbar_arrive(smem_u32(&r.full[slot]));
    }
    w = (int)from_leader((uint32_t)v, lead);
    return true;
}

__device__ __forceinline__ bool sched_take_warp(SchedRing &r, int i, int &w, const Watchdog &wd) {
    const int slot = i & 1;
    const bool ok = mbar_wait(smem_u32(&r.full[slot]), (i >> 1) & 1, wd);
    if (!__all_sync(0xffffffffu, ok)) return false;
    w = r.item[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&r.empty[slot]));
    return true;
}

template <typename T>
__device__ __forceinline__ void zero_cols(T *dst, int n) {
    for (int c = 0; c < n; c += 4) store4(dst + c, make_float4(0.f, 0.f, 0.f, 0.f));
}

// =============================== dK, dV =======================================

struct DkdvInfo {
    int q_start, Lq, k_start, Lk, h, key0, qb0, nq, t;
};

__device__ __forceinline__ DkdvInfo dkdv_info(const BwdParams &p, int w) {
    const WorkItem it = map_item(w, p.sched_kv.prefix, p.n_seq, p.H, false);
    DkdvInfo f;
    seq_bounds(p.cu_q, p.n_q, it.b, f.q_start, f.Lq);
    seq_bounds(p.cu_k, p.n_k, it.b, f.k_start, f.Lk);
    f.h = it.h;
    f.t = it.t;
    f.key0 = it.t * BT;
    f.qb0 = p.causal ? it.t : 0;
    f.nq = max(0, cdiv(f.Lq, BT) - f.qb0);
    return f;
}

struct __align__(8) DkdvBars {
    uint64_t kv_full, kv_empty;
    uint64_t q_full[4], q_empty[4], do_empty[4];  // q_full: the Q and dO tiles of a query block
    uint64_t st_full, dp_full, p_ready, ds_ready, acc_done, acc_free;
    uint64_t stats_ready[2];  // all elementwise threads staged a query block's lse2 / Dr
    uint64_t mma_drain;       // abort path: completion of the MMAs already issued
    uint64_t dq_full, dq_free; // fused dQ: a block's dQ partial is in TMEM / has been read out
    uint64_t dv_done;          // fused dQ: dV of a block has read its dO tile (the slot may take dS)
    SchedRing sched;
};

// Two producer warps, each run by all its 32 lanes in step (uniform waits, one
// elected lane issues the loads): warp 0 publishes the work items and loads K,
// V and the Q ring; warp 2 loads the dO ring.  Splitting them keeps a dO load from waiting
// behind a Q slot (Q tiles are released only after dK, dO tiles after dV).
template <int D>
__device__ void dkdv_producer(const TcBwdArgs &a, DkdvBars &bars, uint32_t sK, uint32_t sV, uint32_t sQ,
                              uint32_t sDO, bool dout_role, const Watchdog &wd) {
    using C = BCfg<D>;
    const BwdParams &p = a.p;
    const int total = p.sched_kv.hdr[1];
    uint32_t kv_uses = 0;
    RingPos<C::kDkdvQStages> qr;
    RingPos<C::kDkdvDoStages> dr;
    bool kv_pending = false;
    // load the Q or dO tile of query block `row` into its ring
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, wd));
    };
    auto load_row = [&](uint64_t *full, uint64_t *empty, uint32_t slot, uint32_t phase, uint32_t base,
                        const CUtensorMap *tm, int row, int h) -> bool {
        if (!wait(empty[slot], phase ^ 1)) return false;
        if (elect_one()) {
            const uint32_t bar = smem_u32(&full[slot]);
            mbar_expect_tx(bar, C::kTileBytes);
#pragma unroll
            for (int g = 0; g < C::kBoxes; ++g)
                tma_load_3d(base + slot * C::kTileBytes + g * C::kBoxBytes, tm, 64 * g, row, h, bar);
        }
        __syncwarp();
        return true;
    };
    for (int i = 0;; ++i) {
        int w;
        if (dout_role) {
            if (!sched_take_warp(bars.sched, i, w, wd)) break;
        } else {
            if (!sched_publish_warp(bars.sched, i, p.sched_kv.hdr, w, wd)) break;
        }
        if (w >= total) break;
        const DkdvInfo f = dkdv_info(p, w);
        if (f.nq == 0) continue;
        bool ok = true;
        if (dout_role) {
            for (int qb = 0; qb < f.nq; ++qb) {
                ok = load_row(bars.q_full, bars.do_empty, dr.slot(), dr.phase(), sDO, &a.tdo,
                              f.q_start + BT * (f.qb0 + qb), f.h);
                if (!ok) break;
                ++dr.i;
            }
            if (!ok) break;
            continue;
        }
        if (!wait(bars.kv_empty, (kv_uses & 1) ^ 1)) break;
        if (elect_one()) {
            const uint32_t bar = smem_u32(&bars.kv_full);
            mbar_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
            for (int g = 0; g < C::kBoxes; ++g) {
                tma_load_3d(sK + g * C::kBoxBytes, &a.tk, 64 * g, f.k_start + f.key0, f.h, bar);
                tma_load_3d(sV + g * C::kBoxBytes, &a.tv, 64 * g, f.k_start + f.key0, f.h, bar);
            }
        }
        __syncwarp();
        ++kv_uses;
        kv_pending = true;
        for (int qb = 0; qb < f.nq; ++qb) {
            ok = load_row(bars.q_full, bars.q_empty, qr.slot(), qr.phase(), sQ, &a.tq,
                          f.q_start + BT * (f.qb0 + qb), f.h);
            if (!ok) break;
            ++qr.i;
        }
        if (!ok) break;
    }
    if (aborting(wd) && (threadIdx.x & 31) == 0) {
        const long long budget = kDrainCycles;  // loads in flight land within microseconds
        for (uint32_t k = qr.i > (uint32_t)C::kDkdvQStages ? qr.i - C::kDkdvQStages : 0; k < qr.i; ++k)
            drain_wait(smem_u32(&bars.q_full[k % C::kDkdvQStages]), (k / C::kDkdvQStages) & 1, budget);
        for (uint32_t k = dr.i > (uint32_t)C::kDkdvDoStages ? dr.i - C::kDkdvDoStages : 0; k < dr.i; ++k)
            drain_wait(smem_u32(&bars.q_full[k % C::kDkdvDoStages]), (k / C::kDkdvDoStages) & 1, budget);
        if (kv_pending) drain_wait(smem_u32(&bars.kv_full), (kv_uses - 1) & 1, budget);
    }
}

template <int D, bool kBF16>
__device__ void dkdv_mma(const TcBwdArgs &a, DkdvBars &bars, uint32_t sK, uint32_t sV, uint32_t sQ, uint32_t sDO,
                         uint32_t tmem, const Watchdog &wd) {
    using C = BCfg<D>;
    const BwdParams &p = a.p;
    const int total = p.sched_kv.hdr[1];
    constexpr uint32_t idSS = idesc_f16(kBF16, BT, BT, 0);
    // S^T with a negative scale: negate K (the A operand) so P uses |scale|
    const uint32_t idST = idSS | (p.scale_log2 < 0.f ? (1u << 13) : 0u);
    constexpr uint32_t idTS = idesc_f16(kBF16, BT, D, 1);
    // Q and dO of a query block share a ring position (one full barrier)
    static_assert(C::kDkdvQStages == C::kDkdvDoStages, "Q and dO rings advance together");
    constexpr uint32_t QS = C::kDkdvQStages;
    uint32_t kv_cnt = 0, af_cnt = 0;

    // Descriptors built once; per MMA a constant is added to the start address.
    const uint64_t kmaj = sdesc_sw128(0, 16, 1024);            // K-major, base address 0
    const uint64_t nmaj = sdesc_sw128(0, C::kBoxBytes, 1024);  // N-major, base address 0
    // (the issue_* lambdas are called by the elected lane)
    // X^T = A B^T with A, B (128 x D) K-major tiles -> TMEM columns [col, col + 128)
    auto issue_ss = [&](uint32_t col, uint32_t A, uint32_t B, uint32_t id) {
        const uint64_t ad = kmaj + sdesc_step(A), bd = kmaj + sdesc_step(B);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = sdesc_step((kk >> 2) * C::kBoxBytes + (kk & 3) * 32);
            mma_ss(tmem + col, ad + off, bd + off, id, kk > 0);
        }
    };
    // acc (+)= X^T Y with X^T 16-bit in TMEM (two 32-column halves at +0 and +64)
    // and Y (128 rows x D) N-major in shared memory
    auto issue_ts = [&](uint32_t acc_col, uint32_t a_col, uint32_t Y, bool acc) {
        const uint64_t yd = nmaj + sdesc_step(Y);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
            mma_ts(tmem + acc_col, tmem + a_col + 8 * kk + (kk >= 4 ? 32 : 0), yd + sdesc_step(kk * 2048), idTS,
                   acc || kk > 0);
    };
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, wd));
    };

    auto due = [](uint64_t &bar, uint32_t parity) { return mbar_due(smem_u32(&bar), parity); };
    // query blocks taken before this item: block b of the item uses Q / dO ring
    // position q0 + b and is phase q0 + b of p_ready and ds_ready
    uint32_t q0 = 0;
    auto qslot = [&](int b) { return (q0 + b) % QS; };
    auto qphase = [&](int b) { return ((q0 + b) / QS) & 1; };

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take_warp(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DkdvInfo f = dkdv_info(p, w);
        if (f.nq == 0) continue;
        if (!wait(bars.kv_full, kv_cnt & 1)) return;
        ++kv_cnt;
        if (!wait(bars.q_full[qslot(0)], qphase(0))) return;  // Q and dO of the block
        tc_fence_after();
        if (elect_one()) {
            issue_ss(0, sK, sQ + qslot(0) * C::kTileBytes, idST);  // S^T = K Q^T
            tc_commit(smem_u32(&bars.st_full));
            issue_ss(BT, sV, sDO + qslot(0) * C::kTileBytes, idSS);  // dP^T = V dO^T
            tc_commit(smem_u32(&bars.dp_full));
        }
        __syncwarp();
        // Per query block qb three issue steps, each behind one barrier:
        //   0: dV += P^T dO           after P^T_qb is in TMEM (p_ready)
        //   1: S^T of block qb + 1    after its Q / dO tiles landed (q_full)
        //   2: dK += dS^T Q, then dP^T of block qb + 1   after dS^T_qb is in TMEM (ds_ready)
        // The elected lane runs the steps back to back, testing each step's
        // barrier (a short spin) while the MMAs before it are still queued, so
        // the tensor pipe does not wait for the warp's own turnaround; only
        // when a barrier is not yet complete does the whole warp wait for it
        // (bounded) and the lane resume from there.
        int qb = 0, step = 0;
        while (qb < f.nq) {
            bool ok;
            if (step == 0) {
                ok = wait(bars.p_ready, (q0 + qb) & 1);
                if (ok && qb == 0) ok = wait(bars.acc_free, (af_cnt & 1) ^ 1);
            } else if (step == 1) {
                ok = wait(bars.q_full[qslot(qb + 1)], qphase(qb + 1));
            } else {
                ok = wait(bars.ds_ready, (q0 + qb) & 1);
            }
            if (!ok) return;
            const bool lead = elect_one();
            if (lead) {
                for (;;) {
                    tc_fence_after();
                    if (step == 0) {
                        issue_ts(256, 0, sDO + qslot(qb) * C::kTileBytes, qb > 0);  // dV += P^T dO
                        tc_commit(smem_u32(&bars.do_empty[qslot(qb)]));
                        step = qb + 1 < f.nq ? 1 : 2;
                    } else if (step == 1) {
                        issue_ss(0, sK, sQ + qslot(qb + 1) * C::kTileBytes, idST);  // S^T of the next block
                        tc_commit(smem_u32(&bars.st_full));
                        step = 2;
                    } else {
                        issue_ts(256 + D, BT, sQ + qslot(qb) * C::kTileBytes, qb > 0);  // dK += dS^T Q
                        tc_commit(smem_u32(&bars.q_empty[qslot(qb)]));
                        if (qb + 1 < f.nq) {
                            issue_ss(BT, sV, sDO + qslot(qb + 1) * C::kTileBytes, idSS);  // dP^T of the next block
                            tc_commit(smem_u32(&bars.dp_full));
                        }
                        ++qb;
                        step = 0;
                    }
                    if (qb == f.nq) break;
                    const bool ready = step == 0   ? due(bars.p_ready, (q0 + qb) & 1)
                                       : step == 1 ? due(bars.q_full[qslot(qb + 1)], qphase(qb + 1))
                                                   : due(bars.ds_ready, (q0 + qb) & 1);
                    if (!ready) break;
                }
            }
            // (block, step) in one word: step < 4 in the low bits, the block
            // index (< 2^24 for 2^31 rows) above them
            const uint32_t st = from_leader(((uint32_t)qb << 2) | (uint32_t)step, lead);
            qb = (int)(st >> 2);
            step = (int)(st & 3u);
        }
        ++af_cnt;
        q0 += f.nq;
        if (elect_one()) {
            tc_commit(smem_u32(&bars.acc_done));
            tc_commit(smem_u32(&bars.kv_empty));
        }
        __syncwarp();
    }
}

// Fused-dQ variant of the issuer: per query block also dQ_qb = dS K, from the
// dS tile the elementwise warps wrote into shared memory (A operand, M-major:
// rows = keys, query rows contiguous) and the resident K tile (B, N-major).
// Issue order S_0, dP_0, then per block dV_qb, dP_qb (qb > 0), S_{qb+1}, dK_qb,
// dQ_qb: the score MMA of the next block covers the elementwise dS work, and
// dV of the next block covers the read-out of dQ_qb.
template <int D, bool kBF16>
__device__ void dkdvq_mma(const TcBwdArgs &a, DkdvBars &bars, uint32_t sK, uint32_t sV, uint32_t sQ,
                          uint32_t sDO, uint32_t sDS, uint32_t tmem, const Watchdog &wd) {
    using C = BCfg<D>;
    const BwdParams &p = a.p;
    const int total = p.sched_kv.hdr[1];
    constexpr uint32_t idSS = idesc_f16(kBF16, BT, BT, 0);
    const uint32_t idST = idSS | (p.scale_log2 < 0.f ? (1u << 13) : 0u);
    constexpr uint32_t idTS = idesc_f16(kBF16, BT, D, 1);
    constexpr uint32_t idDQ = idesc_f16(kBF16, BT, D, 1) | (1u << 15);  // A (dS) M-major
    constexpr bool kAlias = C::kDqCol == (uint32_t)BT;  // dQ shares the dP^T columns
    uint32_t kv_cnt = 0, p_cnt = 0, ds_cnt = 0, af_cnt = 0, dqf_cnt = 0, dq_issued = 0;
    RingPos<C::kDkdvQStages> qr;
    RingPos<C::kDkdvDoStages> dr;

    const uint64_t kmaj = sdesc_sw128(0, 16, 1024);
    const uint64_t nmaj = sdesc_sw128(0, C::kBoxBytes, 1024);
    auto issue_ss = [&](uint32_t col, uint32_t A, uint32_t B, uint32_t id) {
        const uint64_t ad = kmaj + sdesc_step(A), bd = kmaj + sdesc_step(B);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = sdesc_step((kk >> 2) * C::kBoxBytes + (kk & 3) * 32);
            mma_ss(tmem + col, ad + off, bd + off, id, kk > 0);
        }
    };
    auto issue_ts = [&](uint32_t acc_col, uint32_t a_col, uint32_t Y, bool acc) {
        const uint64_t yd = nmaj + sdesc_step(Y);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
            mma_ts(tmem + acc_col, tmem + a_col + 8 * kk + (kk >= 4 ? 32 : 0), yd + sdesc_step(kk * 2048), idTS,
                   acc || kk > 0);
    };
    // dQ = dS K: both operands M/N-major, 128-row slabs of 16 keys 2048 bytes apart
    const uint64_t dsd0 = sdesc_sw128(0, C::kDsBytes / 2, 1024);
    auto issue_dq = [&](uint32_t ds) {
        const uint64_t ad = dsd0 + sdesc_step(ds), bd = nmaj + sdesc_step(sK);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
            mma_ss(tmem + C::kDqCol, ad + sdesc_step(kk * 2048), bd + sdesc_step(kk * 2048), idDQ, kk > 0);
    };
    // every dQ issued so far has been read out of TMEM by the elementwise warps
    auto dq_region_free = [&]() -> bool {
        while (dqf_cnt < dq_issued) {
            if (!mbar_wait(smem_u32(&bars.dq_free), dqf_cnt & 1, wd)) return false;
            ++dqf_cnt;
        }
        return true;
    };
    auto take = [&](uint64_t *full, uint32_t slot, uint32_t phase) -> bool {
        return mbar_wait(smem_u32(&full[slot]), phase, wd);
    };

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DkdvInfo f = dkdv_info(p, w);
        if (f.nq == 0) continue;
        if (!mbar_wait(smem_u32(&bars.kv_full), kv_cnt & 1, wd)) return;
        ++kv_cnt;
        uint32_t qs = qr.slot(), os = dr.slot();
        if (!take(bars.q_full, qs, qr.phase())) return;
        ++qr.i;
        tc_fence_after();
        issue_ss(0, sK, sQ + qs * C::kTileBytes, idST);  // S^T_0 = K Q^T
        tc_commit(smem_u32(&bars.st_full));
        if (kAlias && !dq_region_free()) return;
        ++dr.i;  // dO landed with its Q (q_full)
        tc_fence_after();
        issue_ss(BT, sV, sDO + os * C::kTileBytes, idSS);  // dP^T_0 = V dO^T
        tc_commit(smem_u32(&bars.dp_full));
        for (int qb = 0; qb < f.nq; ++qb) {
            if (qb > 0) {
                os = dr.slot();  // dO landed with its Q (q_full, waited before S^T of this block)
                ++dr.i;
            }
            if (!mbar_wait(smem_u32(&bars.p_ready), p_cnt & 1, wd)) return;
            ++p_cnt;
            if (qb == 0) {
                if (!mbar_wait(smem_u32(&bars.acc_free), (af_cnt & 1) ^ 1, wd)) return;
                ++af_cnt;
            }
            tc_fence_after();
            issue_ts(256, 0, sDO + os * C::kTileBytes, qb > 0);  // dV += P^T dO
            if (C::kDsInDoSlot) tc_commit(smem_u32(&bars.dv_done));
            if (qb > 0) {
                if (kAlias && !dq_region_free()) return;
                tc_fence_after();
                issue_ss(BT, sV, sDO + os * C::kTileBytes, idSS);  // dP^T
                tc_commit(smem_u32(&bars.dp_full));
            }
            uint32_t qsn = 0;
            if (qb + 1 < f.nq) {
                qsn = qr.slot();
                if (!take(bars.q_full, qsn, qr.phase())) return;
                ++qr.i;
                tc_fence_after();
                issue_ss(0, sK, sQ + qsn * C::kTileBytes, idST);  // S^T of the next block
                tc_commit(smem_u32(&bars.st_full));
            }
            if (!mbar_wait(smem_u32(&bars.ds_ready), ds_cnt & 1, wd)) return;
            ++ds_cnt;
            tc_fence_after();
            issue_ts(256 + D, BT, sQ + qs * C::kTileBytes, qb > 0);  // dK += dS^T Q
            tc_commit(smem_u32(&bars.q_empty[qs]));
            if (!kAlias && !dq_region_free()) return;
            tc_fence_after();
            issue_dq(C::kDsInDoSlot ? sDO + os * C::kTileBytes : sDS);  // dQ_qb = dS K
            ++dq_issued;
            tc_commit(smem_u32(&bars.dq_full));
            tc_commit(smem_u32(&bars.do_empty[os]));  // dO, and at D = 128 the dS in its slot
            qs = qsn;
        }
        tc_commit(smem_u32(&bars.acc_done));
        tc_commit(smem_u32(&bars.kv_empty));
    }
}

template <int D, bool kBF16, typename Tg>
__device__ void dkdv_elementwise(const TcBwdArgs &a, DkdvBars &bars, float *stats, uint32_t tmem,
                                 const Watchdog &wd) {
    const BwdParams &p = a.p;
    const int total = p.sched_kv.hdr[1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = threadIdx.x - 128;       // 0..255
    const int wg = (warp - 4) >> 2;        // column half
    const int quarter = warp & 3;
    const int kl = 32 * quarter + lane;    // key row inside the tile = TMEM lane
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    const float sl2 = fabsf(p.scale_log2);  // the score MMA negated S for a negative scale
    uint32_t st_cnt = 0, dp_cnt = 0, ad_cnt = 0, stat_i = 0;

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take_warp(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DkdvInfo f = dkdv_info(p, w);
        const int key = f.key0 + kl;
        const bool live = key < f.Lk;
        Tg *dst = static_cast<Tg *>(wg == 0 ? p.dv : p.dk) +
                  (int64_t)(f.k_start + key) * (wg == 0 ? p.dv_st : p.dk_st) +
                  (int64_t)f.h * (wg == 0 ? p.dv_sh : p.dk_sh);
        if (f.nq == 0) {
            if (live) zero_cols(dst, D);
            continue;
        }
        // lse2 / Dr of a query block, stored negated (the elementwise math adds
        // them); rows past the sequence give P = 0 and Dr = 0.  Each of the 256
        // threads fetches one value one block ahead of its use, from an address
        // clamped into the sequence so that the load needs no predicate and no
        // arithmetic waits on it before the value is staged.
        const float *stat_src = (e < BT ? p.lse2 : p.dr) + (int64_t)f.h * p.n_q + f.q_start;
        auto fetch_stat = [&](int qb, bool &valid) -> float {
            const int qr = BT * (f.qb0 + qb) + (e & (BT - 1));
            valid = qr < f.Lq;
            return __ldg(stat_src + min(qr, f.Lq - 1));
        };
        bool stat_valid;
        float stat_next = fetch_stat(0, stat_valid);
        for (int qb = 0; qb < f.nq; ++qb) {
            float *sb = stats + (stat_i & 1) * 2 * BT;
            sb[e] = stat_valid ? -stat_next : (e < BT ? -INFINITY : 0.f);
            mbar_arrive_warp(smem_u32(&bars.stats_ready[stat_i & 1]));
            bool ok = mbar_wait(smem_u32(&bars.stats_ready[stat_i & 1]), (stat_i >> 1) & 1, wd);
            if (!__all_sync(0xffffffffu, ok)) return;
            ++stat_i;
            if (qb + 1 < f.nq) stat_next = fetch_stat(qb + 1, stat_valid);  // in flight during this block
            const float2 *nlse2 = reinterpret_cast<const float2 *>(sb + 64 * wg);
            const float2 *ndr = reinterpret_cast<const float2 *>(sb + BT + 64 * wg);

            ok = mbar_wait(smem_u32(&bars.st_full), st_cnt & 1, wd);
            ++st_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld_x32(lane_base + 64 * wg, r[0]);
            tmem_ld_x32(lane_base + 64 * wg + 32, r[1]);
            tmem_ld_wait(r[0]);
            tmem_ld_wait(r[1]);
            float2 pr[32];
            const bool diag = p.causal && (f.qb0 + qb == f.t);  // query block == key block
            const float2 sc2 = make_float2(sl2, sl2);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 sv = make_float2(__uint_as_float(r[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(r[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 x = __ffma2_rn(sv, sc2, nlse2[c]);
                const float2 pv = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                pr[c] = pv;
                pk[c] = pack2(pv.x, pv.y, kBF16);
            }
            if (diag) {
                // queries before the key: P^T = 0 (whatever their discarded exponentials
                // gave); kept out of the loop above, which every block runs
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = 64 * wg + 2 * c;
                    if (kl > q + 1) {
                        pr[c] = make_float2(0.f, 0.f);
                        pk[c] = 0u;
                    } else if (kl > q) {
                        pr[c].x = 0.f;
                        pk[c] &= 0xFFFF0000u;  // the pair's first value
                    }
                }
            }
            tmem_st_x32(lane_base + 64 * wg, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.p_ready));

            ok = mbar_wait(smem_u32(&bars.dp_full), dp_cnt & 1, wd);
            ++dp_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            tmem_ld_x32(lane_base + BT + 64 * wg, r[0]);
            tmem_ld_x32(lane_base + BT + 64 * wg + 32, r[1]);
            tmem_ld_wait(r[0]);
            tmem_ld_wait(r[1]);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 dp = make_float2(__uint_as_float(r[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(r[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 d = __fmul2_rn(pr[c], __fadd2_rn(dp, ndr[c]));
                pk[c] = pack2(d.x, d.y, kBF16);
            }
            tmem_st_x32(lane_base + BT + 64 * wg, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.ds_ready));
        }
        // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK * scale
        bool ok = mbar_wait(smem_u32(&bars.acc_done), ad_cnt & 1, wd);
        ++ad_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        const float mul = wg == 0 ? 1.f : p.scale;
        // the warp's 32 key rows: the first one's address, and how many exist
        const int64_t gst = wg == 0 ? p.dv_st : p.dk_st;
        Tg *wrow0 = dst - (int64_t)lane * gst;
        const int rows_live = min(32, max(0, f.Lk - (f.key0 + 32 * quarter)));
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld_x32(lane_base + 256 + D * wg + 32 * c, u);
            tmem_ld_wait(u);
            store_rows_chunk(u, mul, wrow0 + 32 * c, gst, rows_live, lane);
        }
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&bars.acc_free));
    }
}

// Fused-dQ variant of the elementwise warps.  Per query block: P^T (as in the
// separate variant); then the read-out of the previous block's dQ partial from
// TMEM (thread = query row) with f32 reductions into the workspace sums; then
// dS^T, written 16-bit both to TMEM (A operand of dK) and, 128-byte swizzled,
// to shared memory (A operand of dQ).
template <int D, bool kBF16, typename Tg>
__device__ void dkdvq_elementwise(const TcBwdArgs &a, DkdvBars &bars, float *stats, uint32_t sDO, uint32_t sDS,
                                  uint32_t tmem, const Watchdog &wd) {
    using C = BCfg<D>;
    const BwdParams &p = a.p;
    const int total = p.sched_kv.hdr[1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = threadIdx.x - 128;
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int kl = 32 * quarter + lane;    // TMEM lane: key row of S^T / dP^T, query row of dQ
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    const float sl2 = fabsf(p.scale_log2);
    uint32_t st_cnt = 0, dp_cnt = 0, ad_cnt = 0, stat_i = 0, dqf_cnt = 0, blk = 0;
    const int64_t acc_step = (int64_t)p.n_q * 4;  // floats between 4-column groups

    // read dQ of block j of item f out of TMEM and add it to the workspace sums
    auto drain = [&](const DkdvInfo &f, int j) -> bool {
        bool ok = mbar_wait(smem_u32(&bars.dq_full), dqf_cnt & 1, wd);
        ++dqf_cnt;
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc_fence_after();
        const int row = BT * (f.qb0 + j) + kl;
        float *dst = p.dq_accum + (((int64_t)f.h * (D / 4) + wg * (D / 8)) * p.n_q + f.q_start + row) * 4;
        // 32 columns at a time (8 groups of 4); TMEM is released after the last load
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            uint32_t u[32];
            tmem_ld_x32(lane_base + C::kDqCol + (D / 2) * wg + 32 * c, u);
            tmem_ld_wait(u);
            if (c == D / 64 - 1) {
                tc_fence_before();
                mbar_arrive_warp(smem_u32(&bars.dq_free));
            }
            if (row < f.Lq) {
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    red_add_v4(dst + (8 * c + g) * acc_step, __uint_as_float(u[4 * g]), __uint_as_float(u[4 * g + 1]),
                               __uint_as_float(u[4 * g + 2]), __uint_as_float(u[4 * g + 3]));
            }
        }
        return true;
    };

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take_warp(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DkdvInfo f = dkdv_info(p, w);
        const int key = f.key0 + kl;
        const bool live = key < f.Lk;
        Tg *dst = static_cast<Tg *>(wg == 0 ? p.dv : p.dk) +
                  (int64_t)(f.k_start + key) * (wg == 0 ? p.dv_st : p.dk_st) +
                  (int64_t)f.h * (wg == 0 ? p.dv_sh : p.dk_sh);
        if (f.nq == 0) {
            if (live) zero_cols(dst, D);
            continue;
        }
        const float *stat_src = (e < BT ? p.lse2 : p.dr) + (int64_t)f.h * p.n_q + f.q_start;
        auto fetch_stat = [&](int qb, bool &valid) -> float {
            const int qr = BT * (f.qb0 + qb) + (e & (BT - 1));
            valid = qr < f.Lq;
            return __ldg(stat_src + min(qr, f.Lq - 1));
        };
        bool stat_valid;
        float stat_next = fetch_stat(0, stat_valid);
        for (int qb = 0; qb < f.nq; ++qb, ++blk) {
            float *sb = stats + (stat_i & 1) * 2 * BT;
            sb[e] = stat_valid ? -stat_next : (e < BT ? -INFINITY : 0.f);
            mbar_arrive_warp(smem_u32(&bars.stats_ready[stat_i & 1]));
            bool ok = mbar_wait(smem_u32(&bars.stats_ready[stat_i & 1]), (stat_i >> 1) & 1, wd);
            if (!__all_sync(0xffffffffu, ok)) return;
            ++stat_i;
            if (qb + 1 < f.nq) stat_next = fetch_stat(qb + 1, stat_valid);
            const float2 *nlse2 = reinterpret_cast<const float2 *>(sb + 64 * wg);
            const float2 *ndr = reinterpret_cast<const float2 *>(sb + BT + 64 * wg);

            ok = mbar_wait(smem_u32(&bars.st_full), st_cnt & 1, wd);
            ++st_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld_x32(lane_base + 64 * wg, r[0]);
            tmem_ld_x32(lane_base + 64 * wg + 32, r[1]);
            tmem_ld_wait(r[0]);
            tmem_ld_wait(r[1]);
            float2 pr[32];
            const bool diag = p.causal && (f.qb0 + qb == f.t);
            const float2 sc2 = make_float2(sl2, sl2);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 sv = make_float2(__uint_as_float(r[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(r[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 x = __ffma2_rn(sv, sc2, nlse2[c]);
                float2 pv = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                if (!live) {  // key past its sequence (the tile reaches into the next one):
                    pv = make_float2(0.f, 0.f);  // its dS row must add nothing to dQ
                } else if (diag) {
                    if (kl > 64 * wg + 2 * c) pv.x = 0.f;
                    if (kl > 64 * wg + 2 * c + 1) pv.y = 0.f;
                }
                pr[c] = pv;
                pk[c] = pack2(pv.x, pv.y, kBF16);
            }
            tmem_st_x32(lane_base + 64 * wg, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.p_ready));

            if (qb > 0 && !drain(f, qb - 1)) return;

            ok = mbar_wait(smem_u32(&bars.dp_full), dp_cnt & 1, wd);
            ++dp_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            tmem_ld_x32(lane_base + BT + 64 * wg, r[0]);
            tmem_ld_x32(lane_base + BT + 64 * wg + 32, r[1]);
            tmem_ld_wait(r[0]);
            tmem_ld_wait(r[1]);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 dp = make_float2(__uint_as_float(r[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(r[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 d = __fmul2_rn(pr[c], __fadd2_rn(dp, ndr[c]));
                pk[c] = pack2(d.x, d.y, kBF16);
            }
            tmem_st_x32(lane_base + BT + 64 * wg, pk);
            if (C::kDsInDoSlot) {
                // dS goes over this block's dO tile: dV must have read it (dP of
                // the first block of an item is issued before its dV)
                ok = mbar_wait(smem_u32(&bars.dv_done), blk & 1, wd);
                if (!__all_sync(0xffffffffu, ok)) return;
            }
            // the same dS^T row into the shared dS tile: box wg holds query rows
            // [64 wg, 64 wg + 64), 128 bytes per key row, 16-byte chunks swizzled
            const uint32_t ds_row = (C::kDsInDoSlot ? sDO + (blk % C::kDkdvDoStages) * C::kTileBytes : sDS) +
                                    wg * (C::kDsBytes / 2) + kl * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_shared_v4(ds_row + ((j ^ (kl & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.ds_ready));
        }
        if (!drain(f, f.nq - 1)) return;
        bool ok = mbar_wait(smem_u32(&bars.acc_done), ad_cnt & 1, wd);
        ++ad_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        const float mul = wg == 0 ? 1.f : p.scale;
        // the warp's 32 key rows: the first one's address, and how many exist
        const int64_t gst = wg == 0 ? p.dv_st : p.dk_st;
        Tg *wrow0 = dst - (int64_t)lane * gst;
        const int rows_live = min(32, max(0, f.Lk - (f.key0 + 32 * quarter)));
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld_x32(lane_base + 256 + D * wg + 32 * c, u);
            tmem_ld_wait(u);
            store_rows_chunk(u, mul, wrow0 + 32 * c, gst, rows_live, lane);
        }
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&bars.acc_free));
    }
}

template <int D, bool kBF16, typename Tg, bool kFused>
__global__ void __launch_bounds__(kThreads, 1) dkdv_tc_kernel(const __grid_constant__ TcBwdArgs a) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ DkdvBars bars;
    __shared__ __align__(16) float stats[2 * 2 * BT];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sK = base, sV = base + C::kTileBytes, sQ = base + 2 * C::kTileBytes;
    const uint32_t sDO = sQ + C::kDkdvQStages * C::kTileBytes;
    const uint32_t sDS = sDO + C::kDkdvDoStages * C::kTileBytes;  // used at D = 64 only
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Watchdog wd{a.p.watchdog_cycles, &abort_flag, a.p.status};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.kv_full), 1);
        mbar_init(smem_u32(&bars.kv_empty), 1);
        // q_full[s]: one arrival from each producer warp (Q and dO of the same block)
        for (int s = 0; s < C::kDkdvQStages; ++s) {
            mbar_init(smem_u32(&bars.q_full[s]), 2);
            mbar_init(smem_u32(&bars.q_empty[s]), 1);
        }
        for (int s = 0; s < C::kDkdvDoStages; ++s) mbar_init(smem_u32(&bars.do_empty[s]), 1);
        mbar_init(smem_u32(&bars.st_full), 1);
        mbar_init(smem_u32(&bars.dp_full), 1);
        mbar_init(smem_u32(&bars.p_ready), kEw / 32);
        mbar_init(smem_u32(&bars.ds_ready), kEw / 32);
        mbar_init(smem_u32(&bars.acc_done), 1);
        mbar_init(smem_u32(&bars.acc_free), kEw / 32);
        mbar_init(smem_u32(&bars.stats_ready[0]), kEw / 32);
        mbar_init(smem_u32(&bars.stats_ready[1]), kEw / 32);
        mbar_init(smem_u32(&bars.mma_drain), 1);
        mbar_init(smem_u32(&bars.dq_full), 1);
        mbar_init(smem_u32(&bars.dq_free), kEw / 32);
        mbar_init(smem_u32(&bars.dv_done), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars.sched.full[s]), 1);
            mbar_init(smem_u32(&bars.sched.empty[s]), kSchedConsumers + 1);  // + the dO producer
        }
        fence_mbar_init();
        prefetch_tmap(&a.tq);
        prefetch_tmap(&a.tk);
        prefetch_tmap(&a.tv);
        prefetch_tmap(&a.tdo);
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
        regs_dec<kFused ? C::kRegsProducerFused : C::kRegsProducer>();
        if (warp == 0 || warp == 2) dkdv_producer<D>(a, bars, sK, sV, sQ, sDO, warp == 2, wd);  // whole warps
        else if (warp == 1) {
            // the separate issuer runs on the whole warp, the fused one on lane 0
            if constexpr (kFused) {
                if (lane == 0) dkdvq_mma<D, kBF16>(a, bars, sK, sV, sQ, sDO, sDS, tmem, wd);
            } else {
                dkdv_mma<D, kBF16>(a, bars, sK, sV, sQ, sDO, tmem, wd);
            }
            if (lane == 0 && aborting(wd)) {  // let issued MMAs finish before TMEM is freed
                tc_commit(smem_u32(&bars.mma_drain));
                drain_wait(smem_u32(&bars.mma_drain), 0, kDrainCycles);
            }
        }
    } else {
        regs_inc<kFused ? C::kRegsEwFused : C::kRegsEw>();
        if constexpr (kFused) dkdvq_elementwise<D, kBF16, Tg>(a, bars, stats, sDO, sDS, tmem, wd);
        else dkdv_elementwise<D, kBF16, Tg>(a, bars, stats, tmem, wd);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================= dQ =========================================

struct DqInfo {
    int q_start, Lq, k_start, Lk, h, row0, nk;
};

__device__ __forceinline__ DqInfo dq_info(const BwdParams &p, int w) {
    const WorkItem it = map_item(w, p.sched_q.prefix, p.n_seq, p.H, true);
    DqInfo f;
    seq_bounds(p.cu_q, p.n_q, it.b, f.q_start, f.Lq);
    seq_bounds(p.cu_k, p.n_k, it.b, f.k_start, f.Lk);
    f.h = it.h;
    f.row0 = it.t * BT;
    f.nk = p.causal ? cdiv(min(f.Lk, f.row0 + BT), BT) : cdiv(f.Lk, BT);
    return f;
}

struct __align__(8) DqBars {
    uint64_t q_full, q_empty;
    uint64_t k_full[8], k_empty[8], v_empty[8];  // k_full: the K and V tiles of a key block
    // S and dP of a key block are committed, and read out of TMEM, separately:
    // the next block's S starts once every warp has read this block's S, while
    // they still wait for (or read) its dP
    uint64_t s_full, s_free, dp_full, dp_free, acc_done, acc_free;
    // dS of a key block is in TMEM, alternating by block: the next S / dP pair
    // waits only for every warp's read of this one (s_free, dp_free), so a fast warp can
    // finish the next block's dS before a slow one has finished this block's; with
    // one barrier its early arrival would complete the wrong phase
    uint64_t ds_ready[2];
    uint64_t mma_drain;  // abort path: completion of the MMAs already issued
    SchedRing sched;
};

template <int D>
__device__ void dq_producer(const TcBwdArgs &a, DqBars &bars, uint32_t sQ, uint32_t sDO, uint32_t sK, uint32_t sV,
                            const Watchdog &wd) {
    using C = BCfg<D>;
    const BwdParams &p = a.p;
    const int total = p.sched_q.hdr[1];
    uint32_t q_uses = 0;
    RingPos<C::kDqKStages> kr;
    RingPos<C::kDqVStages> vr;
    bool q_pending = false;
    // load the K and V tiles of key block j into their rings; both land on the
    // K slot's full barrier, so the MMA issuer waits once per key block
    auto load_kv = [&](const DqInfo &f, int j) -> bool {
        const uint32_t ks = kr.slot(), vs = vr.slot();
        if (!mbar_wait(smem_u32(&bars.k_empty[ks]), kr.phase() ^ 1, wd)) return false;
        if (!mbar_wait(smem_u32(&bars.v_empty[vs]), vr.phase() ^ 1, wd)) return false;
        const uint32_t bar = smem_u32(&bars.k_full[ks]);
        mbar_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
        for (int g = 0; g < C::kBoxes; ++g) {
            tma_load_3d(sK + ks * C::kTileBytes + g * C::kBoxBytes, &a.tk, 64 * g, f.k_start + BT * j, f.h, bar);
            tma_load_3d(sV + vs * C::kTileBytes + g * C::kBoxBytes, &a.tv, 64 * g, f.k_start + BT * j, f.h, bar);
        }
        ++kr.i;
        ++vr.i;
        return true;
    };
    for (int i = 0;; ++i) {
        int w;
        if (!sched_publish(bars.sched, i, p.sched_q.hdr, w, wd)) break;
        if (w >= total) break;
        const DqInfo f = dq_info(p, w);
        if (f.nk == 0) continue;
        if (!mbar_wait(smem_u32(&bars.q_empty), (q_uses & 1) ^ 1, wd)) break;
        {
            const uint32_t bar = smem_u32(&bars.q_full);
            mbar_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
            for (int g = 0; g < C::kBoxes; ++g) {
                tma_load_3d(sQ + g * C::kBoxBytes, &a.tq, 64 * g, f.q_start + f.row0, f.h, bar);
                tma_load_3d(sDO + g * C::kBoxBytes, &a.tdo, 64 * g, f.q_start + f.row0, f.h, bar);
            }
            ++q_uses;
            q_pending = true;
        }
        bool ok = true;
        for (int j = 0; j < f.nk && ok; ++j) ok = load_kv(f, j);
        if (!ok) break;
    }
    if (aborting(wd)) {
        const long long budget = kDrainCycles;  // loads in flight land within microseconds
        for (uint32_t k = kr.i > (uint32_t)C::kDqKStages ? kr.i - C::kDqKStages : 0; k < kr.i; ++k)
            drain_wait(smem_u32(&bars.k_full[k % C::kDqKStages]), (k / C::kDqKStages) & 1, budget);
        if (q_pending) drain_wait(smem_u32(&bars.q_full), (q_uses - 1) & 1, budget);
    }
}

template <int D, bool kBF16>
__device__ void dq_mma(const TcBwdArgs &a, DqBars &bars, uint32_t sQ, uint32_t sDO, uint32_t sK, uint32_t sV,
                       uint32_t tmem, const Watchdog &wd) {
    using C = BCfg<D>;
    constexpr uint32_t KS = C::kDqKStages, VS = C::kDqVStages;
    const BwdParams &p = a.p;
    const int total = p.sched_q.hdr[1];
    constexpr uint32_t idSS = idesc_f16(kBF16, BT, BT, 0);
    // S with a negative scale: negate Q (the A operand) so P uses |scale|
    const uint32_t idS = idSS | (p.scale_log2 < 0.f ? (1u << 13) : 0u);
    constexpr uint32_t idTS = idesc_f16(kBF16, BT, D, 1);
    uint32_t q_cnt = 0, af_cnt = 0;
    // key blocks taken before this item: block g uses K / V slots g % KS, g % VS,
    // and is the g-th phase of s_free, dp_free and (alternating) ds_ready
    uint32_t g0 = 0;

    const uint64_t kmaj = sdesc_sw128(0, 16, 1024);
    const uint64_t nmaj = sdesc_sw128(0, C::kBoxBytes, 1024);
    const uint64_t dq_desc = kmaj + sdesc_step(sQ), ddo_desc = kmaj + sdesc_step(sDO);
    // one smem x smem contraction over D (the elected lane)
    auto issue_ss = [&](uint32_t col, uint64_t ad, uint32_t B, uint32_t id) {
        const uint64_t bd = kmaj + sdesc_step(B);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + col, sdesc_add(ad, off), sdesc_add(bd, off), id, kk > 0);
        }
    };
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, wd));
    };
    auto due = [](uint64_t &bar, uint32_t parity) { return mbar_due(smem_u32(&bar), parity); };

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take_warp(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DqInfo f = dq_info(p, w);
        if (f.nk == 0) continue;
        if (!wait(bars.q_full, q_cnt & 1)) return;
        ++q_cnt;
        if (!wait(bars.k_full[g0 % KS], (g0 / KS) & 1)) return;
        tc_fence_after();
        if (elect_one()) {
            issue_ss(0, dq_desc, sK + (g0 % KS) * C::kTileBytes, idS);  // S = Q K^T
            tc_commit(smem_u32(&bars.s_full));
            issue_ss(BT, ddo_desc, sV + (g0 % VS) * C::kTileBytes, idSS);  // dP = dO V^T
            tc_commit(smem_u32(&bars.dp_full));
            tc_commit(smem_u32(&bars.v_empty[g0 % VS]));
        }
        __syncwarp();
        // Per key block j (global g = g0 + j) three issue steps, each behind its barriers:
        //   0: S of block j + 1     after every warp has read S_j (s_free) and K / V of j + 1 landed
        //   1: dP of block j + 1    after every warp has read dP_j (dp_free)
        //   2: dQ += dS_j K_j       after dS_j is in TMEM (ds_ready; at j = 0 also acc_free)
        // (steps 0 and 1 of the last block issue nothing but still take their
        // barrier, so that the next item's S and dP overwrite only what was read).
        // The elected lane runs the steps back to back, testing each step's
        // barriers (a short spin) while the MMAs before it are still queued;
        // only when one is not yet complete does the whole warp wait for it
        // (bounded) and the lane resume from there.
        auto ready = [&](int j, int step, bool spin) -> bool {
            const uint32_t g = g0 + j;
            auto chk = [&](uint64_t &bar, uint32_t parity) { return spin ? due(bar, parity) : wait(bar, parity); };
            if (step == 0)
                return chk(bars.s_free, g & 1) &&
                       (j + 1 >= f.nk || chk(bars.k_full[(g + 1) % KS], ((g + 1) / KS) & 1));
            if (step == 1) return chk(bars.dp_free, g & 1);
            return chk(bars.ds_ready[g & 1], (g >> 1) & 1) && (j != 0 || chk(bars.acc_free, (af_cnt & 1) ^ 1));
        };
        int j = 0, step = 0;
        while (j < f.nk) {
            if (!ready(j, step, false)) return;
            const bool lead = elect_one();
            if (lead) {
                for (;;) {
                    const uint32_t g = g0 + j;
                    const bool more = j + 1 < f.nk;
                    tc_fence_after();
                    if (step == 0) {
                        if (more) {
                            issue_ss(0, dq_desc, sK + ((g + 1) % KS) * C::kTileBytes, idS);
                            tc_commit(smem_u32(&bars.s_full));
                        }
                        step = 1;
                    } else if (step == 1) {
                        if (more) {
                            issue_ss(BT, ddo_desc, sV + ((g + 1) % VS) * C::kTileBytes, idSS);
                            tc_commit(smem_u32(&bars.dp_full));
                            tc_commit(smem_u32(&bars.v_empty[(g + 1) % VS]));
                        }
                        step = 2;
                    } else {
                        const uint64_t kd = nmaj + sdesc_step(sK + (g % KS) * C::kTileBytes);
                        const uint32_t ds_col = tmem + 256 + 64 * (j & 1);
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)  // dQ += dS K
                            mma_ts(tmem + 384, ds_col + 8 * kk, sdesc_add(kd, kk * 2048), idTS, j > 0 || kk > 0);
                        tc_commit(smem_u32(&bars.k_empty[g % KS]));
                        ++j;
                        step = 0;
                    }
                    if (j == f.nk || !ready(j, step, true)) break;
                }
            }
            // (block, step) in one word: step < 4 in the low bits, the block
            // index (< 2^24 for 2^31 keys) above them
            const uint32_t st = from_leader(((uint32_t)j << 2) | (uint32_t)step, lead);
            j = (int)(st >> 2);
            step = (int)(st & 3u);
        }
        ++af_cnt;
        g0 += f.nk;
        if (elect_one()) {
            tc_commit(smem_u32(&bars.acc_done));
            tc_commit(smem_u32(&bars.q_empty));
        }
        __syncwarp();
    }
}

template <int D, bool kBF16, typename Tg>
__device__ void dq_elementwise(const TcBwdArgs &a, DqBars &bars, uint32_t tmem, const Watchdog &wd) {
    const BwdParams &p = a.p;
    const int total = p.sched_q.hdr[1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int rl = 32 * quarter + lane;
    const uint32_t lane_base = tmem_addr(tmem, 32 * quarter, 0);
    const float sl2 = fabsf(p.scale_log2);  // the score MMA negated S for a negative scale
    uint32_t s_cnt = 0, dp_cnt = 0, ad_cnt = 0, step = 0;

    for (int i = 0;; ++i) {
        int w;
        if (!sched_take_warp(bars.sched, i, w, wd)) return;
        if (w >= total) return;
        const DqInfo f = dq_info(p, w);
        const int row = f.row0 + rl;
        const bool live = row < f.Lq;
        const int64_t at = (int64_t)f.h * p.n_q + f.q_start + row;
        const float lse2 = live ? p.lse2[at] : INFINITY;
        const float drr = live ? p.dr[at] : 0.f;
        Tg *dst = static_cast<Tg *>(p.dq) + (int64_t)(f.q_start + row) * p.dq_st + (int64_t)f.h * p.dq_sh +
                  (D / 2) * wg;
        if (f.nk == 0) {
            if (live) zero_cols(dst, D / 2);
            continue;
        }
        for (int j = 0; j < f.nk; ++j, ++step) {
            bool ok = mbar_wait(smem_u32(&bars.s_full), s_cnt & 1, wd);
            ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            uint32_t rs[2][32], rp[2][32];
            tmem_ld_x32(lane_base + 64 * wg, rs[0]);
            tmem_ld_x32(lane_base + 64 * wg + 32, rs[1]);
            tmem_ld_wait(rs[0]);
            tmem_ld_wait(rs[1]);
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.s_free));  // the S buffer may be overwritten

            // P = 2^(S scale log2e - lse2), in place of S, while dP may still be in flight
            const float2 sc2 = make_float2(sl2, sl2), nl2 = make_float2(-lse2, -lse2);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                uint32_t &s0 = rs[(2 * c) >> 5][(2 * c) & 31], &s1 = rs[(2 * c + 1) >> 5][(2 * c + 1) & 31];
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(s0), __uint_as_float(s1)), sc2, nl2);
                // all on the SFU: a share of the pairs on the FMA pipe (exp2_fma2)
                // helped while these warps bounded the kernel, but their extra
                // instructions now cost the MMA-issuing warp of the same
                // sub-partition more issue slots than they save (one pair in
                // four: 2.047 ms, one in eight: 2.035, none: 2.007 on the training shape)
                const float2 pv = make_float2(exp2_approx(x.x), exp2_approx(x.y));
                s0 = __float_as_uint(pv.x);
                s1 = __float_as_uint(pv.y);
            }

            ok = mbar_wait(smem_u32(&bars.dp_full), dp_cnt & 1, wd);
            ++dp_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            tmem_ld_x32(lane_base + BT + 64 * wg, rp[0]);
            tmem_ld_x32(lane_base + BT + 64 * wg + 32, rp[1]);
            tmem_ld_wait(rp[0]);
            tmem_ld_wait(rp[1]);
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.dp_free));  // the dP buffer may be overwritten

            const int key0 = BT * j;
            int lim = BT;  // keys [0, lim) of the tile are admitted for this row
            if ((p.causal && key0 + BT - 1 > f.row0) || key0 + BT > f.Lk)
                lim = min(f.Lk - key0, p.causal ? row - key0 + 1 : BT);
            const int c0 = 64 * wg;
            const float2 ndr2 = make_float2(-drr, -drr);
            const bool masked = lim < BT;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 pv = make_float2(__uint_as_float(rs[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(rs[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 dp = make_float2(__uint_as_float(rp[(2 * c) >> 5][(2 * c) & 31]),
                                              __uint_as_float(rp[(2 * c + 1) >> 5][(2 * c + 1) & 31]));
                const float2 d = __fmul2_rn(pv, __fadd2_rn(dp, ndr2));
                pk[c] = pack2(d.x, d.y, kBF16);
            }
            if (masked) {
                // keys at or past lim: dS = 0 (whatever their discarded exponentials
                // gave, inf or NaN included); kept out of the loop above, which
                // every tile runs
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int col = c0 + 2 * c;
                    if (col >= lim) pk[c] = 0u;
                    else if (col + 1 >= lim) pk[c] &= 0xFFFFu;  // the pair's second value
                }
            }
            tmem_st_x32(lane_base + 256 + 64 * (j & 1) + 32 * wg, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.ds_ready[step & 1]));
        }
        bool ok = mbar_wait(smem_u32(&bars.acc_done), ad_cnt & 1, wd);
        ++ad_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        // the warp's 32 query rows: the first one's address, and how many exist
        Tg *wrow0 = dst - (int64_t)lane * p.dq_st;
        const int rows_live = min(32, max(0, f.Lq - (f.row0 + 32 * quarter)));
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
            uint32_t u[32];
            tmem_ld_x32(lane_base + 384 + (D / 2) * wg + 32 * c, u);
            tmem_ld_wait(u);
            store_rows_chunk(u, p.scale, wrow0 + 32 * c, p.dq_st, rows_live, lane);
        }
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&bars.acc_free));
    }
}

template <int D, bool kBF16, typename Tg>
__global__ void __launch_bounds__(kThreads, 1) dq_tc_kernel(const __grid_constant__ TcBwdArgs a) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ DqBars bars;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base, sDO = base + C::kTileBytes, sK = base + 2 * C::kTileBytes;
    const uint32_t sV = sK + C::kDqKStages * C::kTileBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Watchdog wd{a.p.watchdog_cycles, &abort_flag, a.p.status};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bars.q_full), 1);
        mbar_init(smem_u32(&bars.q_empty), 1);
        for (int s = 0; s < C::kDqKStages; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
        }
        for (int s = 0; s < C::kDqVStages; ++s) mbar_init(smem_u32(&bars.v_empty[s]), 1);
        mbar_init(smem_u32(&bars.s_full), 1);
        mbar_init(smem_u32(&bars.dp_full), 1);
        mbar_init(smem_u32(&bars.mma_drain), 1);
        mbar_init(smem_u32(&bars.s_free), kEw / 32);
        mbar_init(smem_u32(&bars.dp_free), kEw / 32);
        mbar_init(smem_u32(&bars.ds_ready[0]), kEw / 32);
        mbar_init(smem_u32(&bars.ds_ready[1]), kEw / 32);
        mbar_init(smem_u32(&bars.acc_done), 1);
        mbar_init(smem_u32(&bars.acc_free), kEw / 32);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars.sched.full[s]), 1);
            mbar_init(smem_u32(&bars.sched.empty[s]), kSchedConsumers);
        }
        fence_mbar_init();
        prefetch_tmap(&a.tq);
        prefetch_tmap(&a.tk);
        prefetch_tmap(&a.tv);
        prefetch_tmap(&a.tdo);
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
        regs_dec<C::kRegsProducer>();
        if (warp == 0 && lane == 0) dq_producer<D>(a, bars, sQ, sDO, sK, sV, wd);
        else if (warp == 1) {
            dq_mma<D, kBF16>(a, bars, sQ, sDO, sK, sV, tmem, wd);  // the whole warp
            if (lane == 0 && aborting(wd)) {  // let issued MMAs finish before TMEM is freed
                tc_commit(smem_u32(&bars.mma_drain));
                drain_wait(smem_u32(&bars.mma_drain), 0, kDrainCycles);
            }
        }
    } else {
        regs_inc<C::kRegsEw>();
        dq_elementwise<D, kBF16, Tg>(a, bars, tmem, wd);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ================================ host ========================================

bool make_maps(const BwdParams &p, TcBwdArgs &a) {
    a.p = p;
    return make_tile_map(&a.tq, p.q, p.dtype, p.D, p.n_q, p.H, p.q_st, p.q_sh) &&
           make_tile_map(&a.tk, p.k, p.dtype, p.D, p.n_k, p.H, p.k_st, p.k_sh) &&
           make_tile_map(&a.tv, p.v, p.dtype, p.D, p.n_k, p.H, p.v_st, p.v_sh) &&
           make_tile_map(&a.tdo, p.dout, p.dtype, p.D, p.n_q, p.H, p.do_st, p.do_sh);
}

template <typename K>
cudaError_t launch(K kern, int smem, const TcBwdArgs &a, int num_ctas, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (num_ctas <= 0) num_ctas = sm_count();
    e = launch_pdl(kern, dim3(num_ctas), dim3(kThreads), smem, s, a);
    count_launch();
    return cudaGetLastError();
}

template <int D, bool kBF16, typename Tg>
cudaError_t launch_typed(const TcBwdArgs &a, int num_ctas, cudaStream_t s, bool dkdv) {
    if (dkdv && a.p.dq_accum)
        return launch(dkdv_tc_kernel<D, kBF16, Tg, true>, BCfg<D>::kDkdvSmem, a, num_ctas, s);
    if (dkdv) return launch(dkdv_tc_kernel<D, kBF16, Tg, false>, BCfg<D>::kDkdvSmem, a, num_ctas, s);
    return launch(dq_tc_kernel<D, kBF16, Tg>, BCfg<D>::kDqSmem, a, num_ctas, s);
}

template <int D>
cudaError_t launch_d(const TcBwdArgs &a, int num_ctas, cudaStream_t s, bool dkdv) {
    const BwdParams &p = a.p;
    if (p.dtype == ATTN_BF16) {
        if (p.grad_dtype == ATTN_F32) return launch_typed<D, true, float>(a, num_ctas, s, dkdv);
        return launch_typed<D, true, __nv_bfloat16>(a, num_ctas, s, dkdv);
    }
    if (p.grad_dtype == ATTN_F32) return launch_typed<D, false, float>(a, num_ctas, s, dkdv);
    return launch_typed<D, false, __half>(a, num_ctas, s, dkdv);
}

cudaError_t launch_bwd(const BwdParams &p, int num_ctas, cudaStream_t s, bool dkdv) {
    TcBwdArgs a;
    if (!make_maps(p, a)) return cudaErrorInvalidValue;
    return p.D == 64 ? launch_d<64>(a, num_ctas, s, dkdv) : launch_d<128>(a, num_ctas, s, dkdv);
}

}  // namespace

bool tc_bwd_supported(const BwdParams &p) {
    if (p.dtype != ATTN_F16 && p.dtype != ATTN_BF16) return false;
    if (p.D != 64 && p.D != 128) return false;
    if (p.n_q <= 0 || p.n_k <= 0) return false;
    return tc_device_ok();
}

int tc_bwd_kv_block(const BwdParams &) { return BT; }
int tc_bwd_q_block(const BwdParams &) { return BT; }

cudaError_t launch_bwd_dkdv_tc(const BwdParams &p, int num_ctas, cudaStream_t s) {
    return launch_bwd(p, num_ctas, s, true);
}

cudaError_t launch_bwd_dq_tc(const BwdParams &p, int num_ctas, cudaStream_t s) {
    return launch_bwd(p, num_ctas, s, false);
}

}  // namespace attn

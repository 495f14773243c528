// Forward attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), for
// f16 / bf16 inputs, D in {64, 128}.
//
// The online-softmax block recurrence of the OCANNL "Module Ir.Online_softmax"
// page (fourth bullet) -- per query row a scan over key blocks carrying the
// running max m and rescaled sum l, the numerator U accumulated with p * v,
// O = U / l after the last block, -inf padding past the sequence end -- mapped
// onto one GB300 SM as follows.
//
// Work item: 256 query rows of one (sequence, head), split in two 128-row
// tiles (t = 0, 1) that ping-pong between the tensor core and the softmax
// warps.  Items are taken from a global counter (persistent grid, one CTA per
// SM) and broadcast to the warp roles through a two-slot shared ring; a single
// sequence whose items fit in one wave runs one item per CTA instead (static
// schedule, no counter, one launch).
//
// Warp roles (12 warps):
//   warp 0      TMA producer: Q tiles, then K_j, V_j tiles into a ring of
//               shared-memory slots (128-byte swizzle, 64-column boxes).
//   warp 1      MMA issuer (the whole warp, one elected lane issuing):
//               S_t = Q_t K_j^T into TMEM, and
//               U_t += P_t V_j with P_t read from TMEM (it overwrites S_t).
//               Issue order PV_j(0), S_{j+1}(0), PV_j(1), S_{j+1}(1) keeps the
//               tensor core busy while the other tile's softmax runs.
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1: thread =
//               query row = TMEM lane.  Loads S (f32) from TMEM, masks the
//               causal diagonal / sequence tail with -inf, updates m and l in
//               the base-2 domain, writes P = 2^(s*scale*log2e - m) as packed
//               16-bit pairs into TMEM, and after the last block normalises
//               U and stores O and lse.
// The row max is refreshed (and U, l rescaled) only when it grows by more than
// 2^8; otherwise the stale max is kept, which leaves O = U / l exact.
//
// TMEM (512 columns): S_0 / P_0 at [0, 128), S_1 / P_1 at [128, 256),
// U_0 at [256, 256 + D), U_1 at [256 + D, 256 + 2D).
//
// Tile pruning (approximate, on request): after S of a 128 x 128 tile is in
// registers the four warps of the tile's softmax warpgroup combine their row
// maxima into the tile's largest score; a tile below the query tile's rolling
// max + log2(rho) is skipped (no exponentials, no value MMA).
//
// Split-K: with n_splits > 1 an item is (256 query rows, key chunk c); both
// tiles scan chunk c of the item's key tiles and write a partial O (f32,
// normalised by its own l) and lse, which a merge kernel combines.
//
// Every mbarrier wait is bounded (sm100::mbar_wait); on expiry the CTA stops
// issuing work, drains its outstanding TMA loads, frees TMEM and exits, and
// the status word reads ATTN_ETIMEOUT.
#include <cfloat>

#include "sm100.cuh"
#include "tc.h"

namespace attn {

namespace {

using namespace sm100;

constexpr int BM = 128;        // query rows per tile (tcgen05 M)
constexpr int BN = 128;        // keys per KV tile
constexpr int NQT = 2;         // query tiles per work item
constexpr int kItemRows = NQT * BM;
constexpr int kThreads = 384;
constexpr int kSchedConsumers = 1 + 8;  // MMA thread + one lane per softmax warp
// Register split: the block is launched at 168 registers per thread (384
// threads); warpgroup 0 (TMA, MMA, two idle warps) gives registers to the two
// softmax warpgroups.  Chosen per D from ptxas spill reports.
constexpr float kRescaleThreshold = 8.f;  // log2 units

// Tunables (compile-time): K and V ring slots at D = 128 (K tiles are released
// after the two score MMAs, V tiles only after the two value MMAs, so V gets the
// deeper ring), and how many exp2 pairs of every ATTN_FWD_EXP_GROUP go to the
// FMA pipe instead of the SFU (0 = none).
#ifndef ATTN_FWD_KSTAGES_D128
#define ATTN_FWD_KSTAGES_D128 2
#endif
#ifndef ATTN_FWD_VSTAGES_D128
#define ATTN_FWD_VSTAGES_D128 3
#endif
#ifndef ATTN_FWD_EXP_GROUP
#define ATTN_FWD_EXP_GROUP 3
#endif
#ifndef ATTN_FWD_EXP_FMA
#define ATTN_FWD_EXP_FMA 0
#endif

// kF8: Q and K are fp8 (e4m3), one byte per element (D = 128 only): their
// tiles are 128 rows x 128 bytes, one 128-byte swizzled box, and the score
// contraction is tcgen05.mma kind::f8f6f4 (K = 32 per instruction); V, P and U
// keep the 16-bit / f32 path.
template <int D, bool kF8 = false>
struct Cfg {
    static_assert(!kF8 || D == 128, "fp8 Q/K: D = 128 only");
    static constexpr int kBoxBytes = 128 * 128;            // one box: 128 rows x 128 bytes
    static constexpr int kVBoxes = D / 64;                  // V: 64 16-bit columns per box
    static constexpr int kVTileBytes = 128 * D * 2;
    static constexpr int kQKBoxes = kF8 ? 1 : D / 64;       // Q / K boxes per tile
    static constexpr int kQKBoxCols = kF8 ? 128 : 64;       // Q / K elements per box row
    static constexpr int kQKTileBytes = kF8 ? 128 * D : kVTileBytes;
    static constexpr int kSSteps = kF8 ? D / 32 : D / 16;   // score MMAs per tile
    static constexpr int kKStages = kF8 ? 4 : (D == 128 ? ATTN_FWD_KSTAGES_D128 : 4);
    static constexpr int kVStages = D == 128 ? ATTN_FWD_VSTAGES_D128 : 4;
    static constexpr int kSmemBytes = (NQT + kKStages) * kQKTileBytes + kVStages * kVTileBytes + 1024;
    static_assert(kSmemBytes + 1024 <= 232448, "shared memory budget (dynamic + static)");
    static constexpr int kRegsProducer = D == 128 ? 88 : 72;
    static constexpr int kRegsSoftmax = D == 128 ? 208 : 216;
    static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * 168, "register split");
};

struct TcFwdArgs {
    CUtensorMap tq, tk, tv;
    FwdParams p;
};

struct __align__(8) FwdBars {
    uint64_t q_full[NQT], q_empty[NQT];
    uint64_t k_full[4], k_empty[4], v_empty[4];  // k_full: the K and V tiles of a key tile
    uint64_t s_full[NQT], p_full[NQT], o_done[NQT], o_free[NQT];
    uint64_t sched_full[2], sched_empty[2];
    uint64_t mma_drain;  // abort path: completion of the MMAs already issued
    uint64_t tile_max[NQT];  // tile pruning: the four warps' row maxima of the tile are in
};

// Tile pruning exchange: per query tile, each softmax warp's largest score of
// the current key tile (double-buffered by use parity), and the decision the
// softmax warps hand to the MMA issuer (1 = pruned: no value MMA).
struct PruneShared {
    float warp_max[NQT][2][4];
    int skip[NQT];
};

struct ItemInfo {
    int q_start, Lq, k_start, Lk, h, row0;
    int c;       // key split (split-K chunk) of this item
    int j0;      // first key tile of the chunk
    int n[NQT];  // key tiles each query tile scans, from j0 on
    int nkv;     // max over the tiles
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Items in the schedule (static: known at launch; dynamic: written by the
// preparation kernel).
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
    // split-K: both query tiles scan the same chunk of the item's key tiles
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

// Bounded wait for outstanding TMA writes before the CTA exits after an abort.
constexpr long long kDrainCycles = 1ll << 31;
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long budget) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) return;
    }
}

// ---- warp 0: TMA producer ------------------------------------------------------
// Run by all 32 lanes of warp 0 in step: uniform waits, one elected lane takes
// the work item and issues the loads (as the MMA issuer, so that the loop's
// arithmetic stays on the uniform datapath beside the busy softmax warps).

template <int D, bool kF8>
__device__ void producer(const TcFwdArgs &a, FwdBars &bars, int *sched_item, uint32_t sQ, uint32_t sK,
                         uint32_t sV, const Watchdog &wd) {
    using C = Cfg<D, kF8>;
    const FwdParams &p = a.p;
    const int total = total_items(p);
    RingPos<C::kKStages> kr;
    RingPos<C::kVStages> vr;
    uint32_t q_uses[NQT] = {0, 0};
    bool q_pending[NQT] = {false, false};
    auto wait = [&](uint64_t &bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar), parity, wd));
    };
    // the K and V tiles of one key tile into their rings; both land on the K
    // slot's full barrier, so the MMA issuer waits once per key tile
    auto load_kv = [&](int row, int h) -> bool {
        const uint32_t ks = kr.slot(), vs = vr.slot();
        if (!wait(bars.k_empty[ks], kr.phase() ^ 1)) return false;
        if (!wait(bars.v_empty[vs], vr.phase() ^ 1)) return false;
        if (elect_one()) {
            const uint32_t bar = smem_u32(&bars.k_full[ks]);
            mbar_expect_tx(bar, C::kQKTileBytes + C::kVTileBytes);
            for (int g = 0; g < C::kQKBoxes; ++g)
                tma_load_3d(sK + ks * C::kQKTileBytes + g * C::kBoxBytes, &a.tk, C::kQKBoxCols * g, row, h, bar);
            for (int g = 0; g < C::kVBoxes; ++g)
                tma_load_3d(sV + vs * C::kVTileBytes + g * C::kBoxBytes, &a.tv, 64 * g, row, h, bar);
        }
        __syncwarp();
        ++kr.i;
        ++vr.i;
        return true;
    };
    for (int i = 0;; ++i) {
        const int slot = i & 1;
        if (!wait(bars.sched_empty[slot], ((i >> 1) & 1) ^ 1)) break;
        int w = 0;
        const bool lead = elect_one();
        if (lead) {
            w = fetch_item(p.sched.hdr, p.static_items, i);
            sched_item[slot] = w;
            mbar_arrive(smem_u32(&bars.sched_full[slot]));
        }
        w = (int)from_leader((uint32_t)w, lead);
        if (w >= total) break;
        const ItemInfo f = item_info(p, w);
        bool ok = true;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
            if (!ok) break;
            if (f.n[t] == 0) continue;
            ok = wait(bars.q_empty[t], (q_uses[t] & 1) ^ 1);
            if (!ok) break;
            if (elect_one()) {
                const uint32_t bar = smem_u32(&bars.q_full[t]);
                mbar_expect_tx(bar, C::kQKTileBytes);
#pragma unroll
                for (int g = 0; g < C::kQKBoxes; ++g)
                    tma_load_3d(sQ + t * C::kQKTileBytes + g * C::kBoxBytes, &a.tq, C::kQKBoxCols * g,
                                f.q_start + f.row0 + BM * t, f.h, bar);
            }
            __syncwarp();
            ++q_uses[t];
            q_pending[t] = true;
        }
        if (!ok) break;
        for (int j = 0; j < f.nkv && ok; ++j) ok = load_kv(f.k_start + BN * (f.j0 + j), f.h);
        if (!ok) break;
    }
    if (aborting(wd) && (threadIdx.x & 31) == 0) {
        // the newest load of every slot may still be landing in shared memory
        const long long budget = kDrainCycles;  // loads in flight land within microseconds
        for (uint32_t k = kr.i > (uint32_t)C::kKStages ? kr.i - C::kKStages : 0; k < kr.i; ++k)
            drain_wait(smem_u32(&bars.k_full[k % C::kKStages]), (k / C::kKStages) & 1, budget);
#pragma unroll
        for (int t = 0; t < NQT; ++t)
            if (q_pending[t]) drain_wait(smem_u32(&bars.q_full[t]), (q_uses[t] - 1) & 1, budget);
    }
}

// ---- warp 1: MMA issuer ----------------------------------------------------------
// Run by all 32 lanes of warp 1 in step: every lane does the same waits (their
// results are the same), and one elected lane issues each group of MMAs and the
// commits.  With the loop converged the compiler keeps the descriptor and
// counter arithmetic on the uniform datapath, so the issue keeps pace even while
// the softmax warps on the same sub-partition fill the FMA and ALU pipes (a
// single lane running the loop alone fell to ~170 cycles per 64-cycle MMA
// beside FMA-bound neighbours in a microbenchmark; converged: ~73).

template <int D, bool kBF16, bool kF8, bool kPrune>
__device__ void mma_issuer(const TcFwdArgs &a, FwdBars &bars, const int *sched_item,
                           const PruneShared *ps, uint32_t sQ, uint32_t sK, uint32_t sV,
                           uint32_t tmem, const Watchdog &wd) {
    using C = Cfg<D, kF8>;
    const FwdParams &p = a.p;
    const int total = total_items(p);
    // a negative scale negates Q in the score MMA (A-negate bit), so the softmax
    // always scales by |scale| (fp8 Q / K take positive scales only)
    const uint32_t idS = kF8 ? idesc_f8(BM, BN)
                             : idesc_f16(kBF16, BM, BN, 0) | (p.scale_log2 < 0.f ? (1u << 13) : 0u);
    constexpr uint32_t idO = idesc_f16(kBF16, BM, D, 1);
    uint32_t q_cnt[NQT] = {0, 0}, p_cnt[NQT] = {0, 0}, of_cnt[NQT] = {0, 0};
    RingPos<C::kKStages> kr;
    RingPos<C::kVStages> vr;

    // Descriptors are built once; per MMA only a constant is added to the start
    // address (issuing must stay faster than the 64-cycle 128x128x16 MMA).
    const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
    const uint64_t k_desc = sdesc_sw128(sK, 16, 1024);
    const uint64_t v_desc = sdesc_sw128(sV, C::kBoxBytes, 1024);
    // S_t = Q_t K^T over D in steps of 32 bytes inside a 128-byte swizzle row
    // (16 elements of a 16-bit type, 32 fp8 elements)
    auto issue_s = [&](int t, uint32_t kslot) {  // K tile in slot `kslot` of the K ring
        const uint64_t qa = q_desc + sdesc_step(t * C::kQKTileBytes);
        const uint64_t ka = k_desc + sdesc_step(kslot * C::kQKTileBytes);
        const uint32_t d = tmem + BN * t;
        if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < C::kSSteps; ++kk) {
                const uint64_t off = sdesc_step((kk >> 2) * C::kBoxBytes + (kk & 3) * 32);
                if (kF8) mma_ss_f8(d, qa + off, ka + off, idS, kk > 0);
                else mma_ss(d, qa + off, ka + off, idS, kk > 0);
            }
            tc_commit(smem_u32(&bars.s_full[t]));
        }
        __syncwarp();
    };
    // U_t (+)= P_t V over the 128 keys in steps of 16 (8 TMEM columns of P)
    auto issue_pv = [&](int t, uint32_t vslot, bool acc) {  // V tile in slot `vslot` of the V ring
        const uint64_t va = v_desc + sdesc_step(vslot * C::kVTileBytes);
        const uint32_t d = tmem + 256 + D * t, pa = tmem + BN * t;
        if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(d, pa + 8 * kk, va + sdesc_step(kk * 2048), idO, acc || kk > 0);
        }
        __syncwarp();
    };
    // the warp's wait: every lane polls (the same observations), and the result
    // is made warp-uniform so that an abort takes all lanes out together
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
        // K_0
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
            const uint32_t vs = vr.slot();  // V_j landed with K_j (k_full, waited before S_j)
            ++vr.i;
            bool have_next_k = false;
            uint32_t nks = 0;
#pragma unroll
            for (int t = 0; t < NQT; ++t) {
                if (j >= f.n[t]) continue;
                if (!wait(bars.p_full[t], p_cnt[t] & 1)) return;
                ++p_cnt[t];
                if (j == 0) {
                    // the previous item's epilogue of this tile has read U_t
                    if (!wait(bars.o_free[t], (of_cnt[t] & 1) ^ 1)) return;
                    ++of_cnt[t];
                }
                tc_fence_after();
                // a pruned tile adds nothing to U (the first tile is always admitted)
                const bool pruned = kPrune && *reinterpret_cast<const volatile int *>(&ps->skip[t]);
                if (!pruned) issue_pv(t, vs, j > 0);
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

// ---- warps 4-11: softmax and epilogue ------------------------------------------

template <int D, bool kBF16, typename Tout, bool kPrune>
__device__ void softmax_wg(const TcFwdArgs &a, FwdBars &bars, const int *sched_item, PruneShared *ps,
                           uint32_t tmem, const Watchdog &wd) {
    const FwdParams &p = a.p;
    const int total = total_items(p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = (warp - 4) >> 2;    // query tile of this warpgroup
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int lrow = 32 * quarter + lane;
    const uint32_t s_addr = tmem_addr(tmem, 32 * quarter, BN * t);
    const uint32_t o_addr = tmem_addr(tmem, 32 * quarter, 256 + D * t);
    // the score MMA negated S when the scale is negative.  Masked scores are -inf
    // before the scale multiplies them; a zero scale is raised to the smallest
    // normal f32 so that they stay -inf (not NaN) while every admitted score
    // still scales to 0 within f32 rounding
    const float sl2 = fmaxf(fabsf(p.scale_log2), FLT_MIN);
    uint32_t s_cnt = 0, o_cnt = 0, tm_cnt = 0;
    Tout *go = static_cast<Tout *>(p.o);

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
        const int row = r0 + lrow;  // query offset inside the sequence
        Tout *orow = go + f.c * p.o_split_st + (int64_t)(f.q_start + row) * p.o_st + (int64_t)f.h * p.o_sh;
        float *lse_at = p.lse ? p.lse + f.c * p.lse_split_st + (int64_t)f.h * p.n_q + f.q_start + row : nullptr;
        if (n == 0) {
            // rows of this tile exist but admit no key (empty key sequence, or
            // a key split past the tile's last key tile)
            if (r0 < f.Lq && row < f.Lq) {
#pragma unroll 4
                for (int c = 0; c < D; c += 4) store4(orow + c, make_float4(0.f, 0.f, 0.f, 0.f));
                if (lse_at) *lse_at = -INFINITY;
            }
            continue;
        }

        float m = -INFINITY, l = 0.f;
        float m_run = -INFINITY;  // tile pruning: largest score of the admitted tiles (log2 units)
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(smem_u32(&bars.s_full[t]), s_cnt & 1, wd);
            ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_x32(s_addr + 32 * c, r[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(r[c]);
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(r[c >> 5][c & 31]);

            const int key0 = BN * (f.j0 + j);
            const bool masked = (p.causal && key0 + BN - 1 > r0) || key0 + BN > f.Lk;
            if (masked) {
                const int lim = min(f.Lk - key0, p.causal ? row - key0 + 1 : BN);  // keys [0, lim) admitted
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= lim) s[c] = -INFINITY;
            }
            const float mx = row_max<BN>(s) * sl2;
            if (kPrune) {
                // largest score of the whole 128 x 128 tile (rows past the queries excluded),
                // gathered from the four warps through shared memory and an mbarrier
                float tm = row < f.Lq ? mx : -INFINITY;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
                const int par = tm_cnt & 1;
                if (lane == 0) {
                    ps->warp_max[t][par][quarter] = tm;
                    mbar_arrive(smem_u32(&bars.tile_max[t]));
                }
                ok = mbar_wait(smem_u32(&bars.tile_max[t]), par, wd);
                ++tm_cnt;
                if (!__all_sync(0xffffffffu, ok)) return;
                const volatile float *wm = ps->warp_max[t][par];
                const float m_tile = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
                const bool admit = m_run == -INFINITY || m_tile >= m_run + p.prune_log2;
                if (lrow == 0) *reinterpret_cast<volatile int *>(&ps->skip[t]) = admit ? 0 : 1;
                if (!admit) {
                    // nothing of this tile enters m, l or U; S_t may be overwritten
                    if (lrow == 0 && p.pruned_tiles) atomicAdd(p.pruned_tiles, 1ull);
                    tc_fence_before();
                    mbar_arrive_warp(smem_u32(&bars.p_full[t]));
                    continue;
                }
                m_run = fmaxf(m_run, m_tile);
            }
            const float m_new = fmaxf(m, mx);
            // refresh the max only when it grew by more than 2^8 somewhere in the warp
            const bool rescale = j > 0 && __any_sync(0xffffffffu, m_new > m + kRescaleThreshold);
            float alpha = 1.f;
            if (j == 0) {
                m = m_new;
            } else if (rescale) {
                alpha = exp2_approx(m - m_new);
                m = m_new;
            }
            const float m_use = m == -INFINITY ? 0.f : m;
            // p = 2^(s * scale * log2e - m): packed FMA pairs, four packed partial sums
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 x = __ffma2_rn(make_float2(s[64 * hh + 2 * e], s[64 * hh + 2 * e + 1]), sc2, nm2);
                    // optionally some pairs on the FMA pipe (unmasked tiles), the rest on the SFU
                    const bool on_fma = ATTN_FWD_EXP_FMA > 0 && !masked &&
                                        (e % ATTN_FWD_EXP_GROUP) < ATTN_FWD_EXP_FMA;
                    const float2 pv = on_fma ? exp2_fma2(x) : make_float2(exp2_approx(x.x), exp2_approx(x.y));
                    acc[e & 3] = __fadd2_rn(acc[e & 3], pv);
                    pk[e] = pack2(pv.x, pv.y, kBF16);
                }
                tmem_st_x32(s_addr + 32 * hh, pk);
            }
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a03 = __fadd2_rn(a01, a23);
            const float sum = a03.x + a03.y;
            l = l * alpha + sum;
            if (rescale) {
                // U_t is stable here: S_j(t) completed after PV_{j-1}(t)
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t u[32];
                    tmem_ld_x32(o_addr + 32 * c, u);
                    tmem_ld_wait(u);
#pragma unroll
                    for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                    tmem_st_x32(o_addr + 32 * c, u);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&bars.p_full[t]));
        }

        // epilogue: O = U / l, lse = (m + log2 l) ln 2
        ok = mbar_wait(smem_u32(&bars.o_done[t]), o_cnt & 1, wd);
        ++o_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool live = row < f.Lq;
        // the warp's 32 rows: the first one's address, and how many exist
        Tout *wrow0 = go + f.c * p.o_split_st + (int64_t)(f.q_start + r0 + 32 * quarter) * p.o_st +
                      (int64_t)f.h * p.o_sh;
        const int rows_live = min(32, max(0, f.Lq - (r0 + 32 * quarter)));
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld_x32(o_addr + 32 * c, u);
            tmem_ld_wait(u);
            store_rows_chunk(u, inv, wrow0 + 32 * c, p.o_st, rows_live, lane);
        }
        if (live && lse_at) *lse_at = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&bars.o_free[t]));
    }
}

// kPrune: the tile-pruned forward (its tile-max exchange is compiled only there)
template <int D, bool kBF16, typename Tout, bool kF8, bool kPrune>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcFwdArgs a) {
    using C = Cfg<D, kF8>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ FwdBars bars;
    __shared__ PruneShared prune_shared;
    __shared__ int sched_item[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;
    const uint32_t sK = sQ + NQT * C::kQKTileBytes;
    const uint32_t sV = sK + C::kKStages * C::kQKTileBytes;
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
            mbar_init(smem_u32(&bars.tile_max[t]), 4);
        }
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(smem_u32(&bars.k_full[s]), 1);
            mbar_init(smem_u32(&bars.k_empty[s]), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) mbar_init(smem_u32(&bars.v_empty[s]), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars.sched_full[s]), 1);
            mbar_init(smem_u32(&bars.sched_empty[s]), kSchedConsumers);
        }
        mbar_init(smem_u32(&bars.mma_drain), 1);
        fence_mbar_init();
        prefetch_tmap(&a.tq);
        prefetch_tmap(&a.tk);
        prefetch_tmap(&a.tv);
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
        if (warp == 0) {
            producer<D, kF8>(a, bars, sched_item, sQ, sK, sV, wd);  // the whole warp
        } else if (warp == 1) {
            mma_issuer<D, kBF16, kF8, kPrune>(a, bars, sched_item, &prune_shared, sQ, sK, sV, tmem, wd);
            if (lane == 0 && aborting(wd)) {  // let issued MMAs finish before TMEM is freed
                tc_commit(smem_u32(&bars.mma_drain));
                drain_wait(smem_u32(&bars.mma_drain), 0, kDrainCycles);
            }
        }
    } else {
        regs_inc<C::kRegsSoftmax>();
        softmax_wg<D, kBF16, Tout, kPrune>(a, bars, sched_item, &prune_shared, tmem, wd);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- host side ------------------------------------------------------------------

template <int D, bool kBF16, typename Tout, bool kF8>
cudaError_t launch_typed(const TcFwdArgs &args, int num_ctas, cudaStream_t s) {
    auto kern = args.p.prune ? fwd_tc_kernel<D, kBF16, Tout, kF8, true> : fwd_tc_kernel<D, kBF16, Tout, kF8, false>;
    const int smem = Cfg<D, kF8>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (num_ctas <= 0) num_ctas = sm_count();
    e = launch_pdl(kern, dim3(num_ctas), dim3(kThreads), smem, s, args);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, bool kF8>
cudaError_t launch_d(const TcFwdArgs &args, int num_ctas, cudaStream_t s) {
    const FwdParams &p = args.p;
    if (p.dtype == ATTN_BF16) {
        if (p.o_dtype == ATTN_F32) return launch_typed<D, true, float, kF8>(args, num_ctas, s);
        return launch_typed<D, true, __nv_bfloat16, kF8>(args, num_ctas, s);
    }
    if (p.o_dtype == ATTN_F32) return launch_typed<D, false, float, kF8>(args, num_ctas, s);
    return launch_typed<D, false, __half, kF8>(args, num_ctas, s);
}

}  // namespace

bool tc_fwd_supported(const FwdParams &p) {
    if (p.dtype == ATTN_F32) return x3_fwd_supported(p);
    if (p.dtype != ATTN_F16 && p.dtype != ATTN_BF16) return false;
    if (p.D != 64 && p.D != 128) return false;
    if (p.qk_fp8 && (p.D != 128 || !(p.scale_log2 > 0.f))) return false;
    if (p.n_q <= 0 || p.n_k <= 0) return false;
    return tc_device_ok();
}

int tc_fwd_block_rows(const FwdParams &) { return kItemRows; }

cudaError_t launch_fwd_tc(const FwdParams &p, int num_ctas, cudaStream_t s) {
    if (p.dtype == ATTN_F32) return launch_fwd_x3(p, num_ctas, s);
    TcFwdArgs args;
    args.p = p;
    const int qk_dtype = p.qk_fp8 ? kDtypeE4M3 : p.dtype;
    if (!make_tile_map(&args.tq, p.q, qk_dtype, p.D, p.n_q, p.H, p.q_st, p.q_sh) ||
        !make_tile_map(&args.tk, p.k, qk_dtype, p.D, p.n_k, p.H, p.k_st, p.k_sh) ||
        !make_tile_map(&args.tv, p.v, p.dtype, p.D, p.n_k, p.H, p.v_st, p.v_sh))
        return cudaErrorInvalidValue;
    if (p.qk_fp8) return p.D == 128 ? launch_d<128, true>(args, num_ctas, s) : cudaErrorInvalidValue;
    return p.D == 64 ? launch_d<64, false>(args, num_ctas, s) : launch_d<128, false>(args, num_ctas, s);
}

}  // namespace attn

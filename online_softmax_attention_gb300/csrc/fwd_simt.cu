// Forward attention on CUDA cores (FP32 FFMA), any input dtype.
//
// This is the f32-accurate path (f32 inputs are never rounded to a narrower
// type) and the portable path for f16/bf16.  It runs the online-softmax block
// recurrence of the OCANNL "Module Ir.Online_softmax" page (fourth bullet):
// per query tile of 64 rows, a scan over key tiles of 64 keys keeps the row
// max m and the rescaled sum l, accumulates U = sum p * v, and writes
// O = U / l and lse = m + ln l after the last tile.  Keys past the end of the
// sequence, and keys j > i under the causal relation, score -inf (the guarded
// tail).  Scores are kept in the base-2 domain (s * scale * log2 e).
//
// Split-K: with n_splits > 1 every query tile is n_splits work items, each
// scanning one contiguous chunk of the tile's key tiles and writing its own
// partial O (f32, normalised by its own l) and lse; a merge kernel combines them.
//
// Layout: 256 threads; thread (ty, tx) = (tid / 16, tid % 16) owns query rows
// ty + 16 r and keys tx + 16 c (r, c < 4) of the score tile, and output
// columns 64 g + 4 tx + e of its four rows.  Tiles are staged in shared memory
// as f32 rows padded to D + 4 floats, which makes the 16-byte reads of a
// quarter warp fall on distinct banks.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

namespace {

constexpr int BQ = kSimtBlock;  // query rows per work item
constexpr int BK = 64;          // keys per tile
constexpr int NT = 256;
constexpr int LDP = BK + 4;

// f32 inputs at D = 64 stage K and V with cp.async into two alternating
// buffers, so the next key tile's loads overlap this tile's arithmetic (two
// CTAs per SM still fit); other cases stage synchronously through registers.
template <typename Tin, int D>
constexpr bool kAsyncKV = sizeof(Tin) == 4 && D == 64;

// The score contraction uses packed FP32 FMAs (fma.rn.f32x2: two FMAs per
// instruction), pairing adjacent d into separate even / odd partial sums, so
// each operand pair is two adjacent registers of a 16-byte shared-memory load
// of a Q or K row.  (Pairing keys in the value contraction the same way needs V
// key-pair interleaved in shared memory; with the extra repacking pass and
// barrier that was slower, 158 vs 150 us at the cross f32 8192 x 2048 shape.)

template <typename Tin, int D>
constexpr size_t fwd_smem_bytes() {
    return sizeof(float) * (size_t)(BQ * (D + 4) + (kAsyncKV<Tin, D> ? 4 : 2) * BK * (D + 4) + BQ * LDP);
}

// Start copying rows [row0, row0 + 64) of an f32 (tokens, heads, D) tensor
// into shared memory (16-byte cp.async per chunk; rows at or beyond `nrows`
// are zero-filled without reading global memory).
template <int D>
__device__ __forceinline__ void stage_tile_async(float *dst, const float *src, int64_t st, int row0,
                                                 int nrows) {
    constexpr int LD = D + 4;
    constexpr int CPR = D / 4;
    for (int c = threadIdx.x; c < 64 * CPR; c += NT) {
        const int r = c / CPR, cc = c - r * CPR;
        const bool in = row0 + r < nrows;
        const float *g = in ? src + (int64_t)(row0 + r) * st + cc * 4 : src;
        const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(dst + r * LD + cc * 4));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(g), "r"(in ? 16 : 0)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most `n` (0 or 2: the next tile's K and V groups) of this
// thread's cp.async groups are still pending.
__device__ __forceinline__ void cp_async_wait_all_but(int n) {
    if (n == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
    else asm volatile("cp.async.wait_group 2;" ::: "memory");
}

// Stage rows [row0, row0 + 64) of a (tokens, heads, D) tensor into shared
// memory as f32; rows at or beyond `nrows` are zero.
template <typename T, int D>
__device__ __forceinline__ void stage_tile(float *dst, const T *src, int64_t st, int row0,
                                           int nrows) {
    constexpr int LD = D + 4;
    constexpr int CPR = D / 4;  // 4-element chunks per row
    for (int c = threadIdx.x; c < 64 * CPR; c += NT) {
        const int r = c / CPR, cc = c - r * CPR;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < nrows) x = load4(src + (int64_t)(row0 + r) * st + cc * 4);
        *reinterpret_cast<float4 *>(dst + r * LD + cc * 4) = x;
    }
}

template <typename Tin, typename Tout, int D>
__global__ void __launch_bounds__(NT) fwd_simt_kernel(const FwdParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int LD = D + 4;
    constexpr int NG = D / 64;  // column groups of 64 per thread row
    constexpr bool kAsync = kAsyncKV<Tin, D>;
    extern __shared__ float4 smem4[];
    float *sQ = reinterpret_cast<float *>(smem4);
    float *sKb = sQ + BQ * LD;                        // K buffer(s), then V buffer(s)
    float *sVb = sKb + (kAsync ? 2 : 1) * BK * LD;
    float *sP = sVb + (kAsync ? 2 : 1) * BK * LD;
    __shared__ int s_w;
    __shared__ float s_tile_max[NT / 32];  // tile pruning: per-warp largest score

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int total = p.static_items > 0 ? p.static_items : p.sched.hdr[1];
    const Tin *gq = static_cast<const Tin *>(p.q);
    const Tin *gk = static_cast<const Tin *>(p.k);
    const Tin *gv = static_cast<const Tin *>(p.v);
    Tout *go = static_cast<Tout *>(p.o);

    for (int fetch = 0;; ++fetch) {
        if (tid == 0) s_w = fetch_item(p.sched.hdr, p.static_items, fetch);
        __syncthreads();
        const int w = s_w;
        __syncthreads();
        if (w >= total) break;
        const WorkItem it = p.static_items > 0 ? map_item_single(w, p.static_items, p.H, true, p.n_splits)
                                               : map_item(w, p.sched.prefix, p.n_seq, p.H, true, p.n_splits);
        int q_start, Lq, k_start, Lk;
        seq_bounds(p.cu_q, p.n_q, it.b, q_start, Lq);
        seq_bounds(p.cu_k, p.n_k, it.b, k_start, Lk);
        const int row0 = it.t * BQ;
        const int h = it.h;

        stage_tile<Tin, D>(sQ, gq + (int64_t)q_start * p.q_st + (int64_t)h * p.q_sh, p.q_st, row0, Lq);

        float m[4], l[4], acc[4][NG * 4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < NG * 4; ++e) acc[r][e] = 0.f;
        }
        const int n_keys = p.causal ? min(Lk, row0 + BQ) : Lk;
        // split-K: this item scans chunk it.c of the row's key tiles
        const KeyChunk chunk = key_chunk((n_keys + BK - 1) / BK, p.n_splits, it.c);
        float m_run = -INFINITY;  // tile pruning: largest score of the admitted tiles (log2 units)
        const Tin *kbase = gk + (int64_t)k_start * p.k_st + (int64_t)h * p.k_sh;
        const Tin *vbase = gv + (int64_t)k_start * p.v_st + (int64_t)h * p.v_sh;

        if constexpr (kAsync) {
            if (chunk.begin < chunk.end) {
                __syncthreads();  // the previous item's last tile is no longer read
                stage_tile_async<D>(sKb, reinterpret_cast<const float *>(kbase), p.k_st, chunk.begin * BK, Lk);
                stage_tile_async<D>(sVb, reinterpret_cast<const float *>(vbase), p.v_st, chunk.begin * BK, Lk);
            }
        }
        for (int kt = chunk.begin; kt < chunk.end; ++kt) {
            const int key0 = kt * BK;
            __syncthreads();  // previous tile's sK / sV / sP no longer read
            float *sK = sKb, *sV = sVb;
            if constexpr (kAsync) {
                const int buf = (kt - chunk.begin) & 1;
                sK = sKb + buf * BK * LD;
                sV = sVb + buf * BK * LD;
                const bool more = kt + 1 < chunk.end;
                if (more) {  // the next tile into the other buffer, read two iterations ago
                    float *nK = sKb + (buf ^ 1) * BK * LD, *nV = sVb + (buf ^ 1) * BK * LD;
                    stage_tile_async<D>(nK, reinterpret_cast<const float *>(kbase), p.k_st, key0 + BK, Lk);
                    stage_tile_async<D>(nV, reinterpret_cast<const float *>(vbase), p.v_st, key0 + BK, Lk);
                }
                cp_async_wait_all_but(more ? 2 : 0);  // this tile's two groups have landed
            } else {
                stage_tile<Tin, D>(sK, kbase, p.k_st, key0, Lk);
                stage_tile<Tin, D>(sV, vbase, p.v_st, key0, Lk);
            }
            __syncthreads();

            // score micro-tile: rows ty + 16 r, keys tx + 16 c; packed FMAs over
            // (d, d + 1) pairs into even / odd partial sums
            float s[4][4];
            {
                float2 s2[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) s2[r][c] = make_float2(0.f, 0.f);
                // (unrolled by 2: deeper unrolling spills under the 128-register cap)
#pragma unroll 2
                for (int d = 0; d < D; d += 4) {
                    float4 b[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) b[c] = *reinterpret_cast<const float4 *>(sK + (tx + 16 * c) * LD + d);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float4 a = *reinterpret_cast<const float4 *>(sQ + (ty + 16 * r) * LD + d);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            s2[r][c] = __ffma2_rn(make_float2(a.x, a.y), make_float2(b[c].x, b[c].y), s2[r][c]);
                            s2[r][c] = __ffma2_rn(make_float2(a.z, a.w), make_float2(b[c].z, b[c].w), s2[r][c]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) s[r][c] = s2[r][c].x + s2[r][c].y;
            }

            // scale into the base-2 domain, mask
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = row0 + ty + 16 * r;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int key = key0 + tx + 16 * c;
                    const bool ok = key < Lk && (!p.causal || key <= row);
                    s[r][c] = ok ? s[r][c] * p.scale_log2 : -INFINITY;
                }
            }
            if (p.prune) {
                // tile pruning: the largest score of the 64 x 64 tile (rows past the
                // queries excluded) against the query tile's rolling max
                float tm = -INFINITY;
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (row0 + ty + 16 * r < Lq)
#pragma unroll
                        for (int c = 0; c < 4; ++c) tm = fmaxf(tm, s[r][c]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
                if ((tid & 31) == 0) s_tile_max[tid >> 5] = tm;
                __syncthreads();
                float m_tile = s_tile_max[0];
#pragma unroll
                for (int w8 = 1; w8 < NT / 32; ++w8) m_tile = fmaxf(m_tile, s_tile_max[w8]);
                const bool admit = m_run == -INFINITY || m_tile >= m_run + p.prune_log2;
                if (!admit) {  // uniform across the block: nothing of this tile is used
                    if (tid == 0 && p.pruned_tiles) atomicAdd(p.pruned_tiles, 1ull);
                    continue;   // the next tile's first barrier orders the s_tile_max reuse
                }
                m_run = fmaxf(m_run, m_tile);
            }
            // online softmax update
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) mx = fmaxf(mx, s[r][c]);
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_new = fmaxf(m[r], mx);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // row with nothing admitted yet
                const float alpha = exp2_approx(m[r] - m_use);
                float rs = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float pv = exp2_approx(s[r][c] - m_use);
                    rs += pv;
                    sP[(ty + 16 * r) * LDP + tx + 16 * c] = pv;
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
                l[r] = alpha * l[r] + rs;
                m[r] = m_new;
#pragma unroll
                for (int e = 0; e < NG * 4; ++e) acc[r][e] *= alpha;
            }
            __syncthreads();

            // U += P V
#pragma unroll 2
            for (int j = 0; j < BK; j += 4) {
                float4 pr[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) pr[r] = *reinterpret_cast<const float4 *>(sP + (ty + 16 * r) * LDP + j);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const float4 vv = *reinterpret_cast<const float4 *>(sV + (j + jj) * LD + 64 * g + 4 * tx);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float pj = jj == 0 ? pr[r].x : jj == 1 ? pr[r].y : jj == 2 ? pr[r].z : pr[r].w;
                            acc[r][4 * g + 0] = fmaf(pj, vv.x, acc[r][4 * g + 0]);
                            acc[r][4 * g + 1] = fmaf(pj, vv.y, acc[r][4 * g + 1]);
                            acc[r][4 * g + 2] = fmaf(pj, vv.z, acc[r][4 * g + 2]);
                            acc[r][4 * g + 3] = fmaf(pj, vv.w, acc[r][4 * g + 3]);
                        }
                    }
                }
            }
        }

        // epilogue: O = U / l, lse = m ln 2 + ln l
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + ty + 16 * r;
            if (row >= Lq) continue;
            const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
            Tout *orow = go + it.c * p.o_split_st + (int64_t)(q_start + row) * p.o_st + (int64_t)h * p.o_sh;
#pragma unroll
            for (int g = 0; g < NG; ++g)
                store4(orow + 64 * g + 4 * tx,
                       make_float4(acc[r][4 * g] * inv, acc[r][4 * g + 1] * inv,
                                   acc[r][4 * g + 2] * inv, acc[r][4 * g + 3] * inv));
            if (tx == 0 && p.lse)
                p.lse[it.c * p.lse_split_st + (int64_t)h * p.n_q + q_start + row] =
                    l[r] > 0.f ? m[r] * kLn2 + logf(l[r]) : -INFINITY;
        }
    }
}

// Launches the kernel (num_ctas >= 0), or with num_ctas < 0 only reports its
// resident CTAs per SM through *per_sm_out.
template <typename Tin, typename Tout, int D>
cudaError_t launch_typed(const FwdParams &p, int num_ctas, cudaStream_t s, int *per_sm_out) {
    auto kern = fwd_simt_kernel<Tin, Tout, D>;
    const size_t smem = fwd_smem_bytes<Tin, D>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (num_ctas <= 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
        if (e != cudaSuccess) return e;
        if (num_ctas < 0) {
            *per_sm_out = per_sm > 0 ? per_sm : 1;
            return cudaSuccess;
        }
        num_ctas = sm_count() * (per_sm > 0 ? per_sm : 1);
    }
    e = launch_pdl(kern, dim3(num_ctas), dim3(NT), smem, s, p);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tin, int D>
cudaError_t launch_out(const FwdParams &p, int num_ctas, cudaStream_t s, int *per_sm) {
    if (p.o_dtype == ATTN_F32) return launch_typed<Tin, float, D>(p, num_ctas, s, per_sm);
    return launch_typed<Tin, Tin, D>(p, num_ctas, s, per_sm);
}

template <int D>
cudaError_t launch_d(const FwdParams &p, int num_ctas, cudaStream_t s, int *per_sm) {
    switch (p.dtype) {
    case ATTN_F16: return launch_out<__half, D>(p, num_ctas, s, per_sm);
    case ATTN_BF16: return launch_out<__nv_bfloat16, D>(p, num_ctas, s, per_sm);
    default: return launch_typed<float, float, D>(p, num_ctas, s, per_sm);
    }
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdParams &p, int num_ctas, cudaStream_t s) {
    if (num_ctas < 0) num_ctas = 0;
    return p.D == 64 ? launch_d<64>(p, num_ctas, s, nullptr) : launch_d<128>(p, num_ctas, s, nullptr);
}

int fwd_simt_ctas_per_sm(const FwdParams &p) {
    int per_sm = 1;
    // the split-K pass stores f32 partials: ask about that kernel instance
    FwdParams q = p;
    q.o_dtype = ATTN_F32;
    const cudaError_t e = q.D == 64 ? launch_d<64>(q, -1, nullptr, &per_sm) : launch_d<128>(q, -1, nullptr, &per_sm);
    return e == cudaSuccess ? per_sm : 1;
}

}  // namespace attn

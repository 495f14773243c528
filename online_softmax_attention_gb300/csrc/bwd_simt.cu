// Backward attention on CUDA cores (FP32 FFMA), any input dtype, and the
// row-dot preprocessing shared by every backward path.
//
// The fused backward of the OCANNL "Module Ir.Online_softmax" page (third
// bullet) replaces every (seq, seq) gradient buffer with a per-row
// Dr = sum(dO * O) and nests that recompute each pair's p, dp and
// ds = p * (dp - Dr): one over the keys accumulating dk and dv, one over the
// query rows accumulating dq, each owning what it writes.  Here:
//   preprocess  Dr_i = <dO_i, O_i> (f32) and lse2_i = lse_i * log2(e), one warp
//               per (row, head);
//   dkdv        one work item per (sequence, head, 64-key block): loop over the
//               64-row query blocks that can see the block, recompute
//               P = 2^(s*scale*log2e - lse*log2e), dV += P^T dO, dP = dO V^T,
//               dS = P (dP - Dr), dK += dS^T Q; write dK * scale and dV once;
//   dq          one work item per (sequence, head, 64-row query block): loop
//               over key blocks, recompute P, dP, dS; dQ += dS K; write
//               dQ * scale once.
// Thread layout and shared-memory padding follow the SIMT forward kernel.
#include "../../include/attn.h"
#include "common.cuh"

namespace attn {

namespace {

constexpr int B = kSimtBlock;  // rows per query block = keys per key block
constexpr int NT = 256;
constexpr int LDP = B + 4;

template <typename T, int D>
__device__ __forceinline__ void stage_tile(float *dst, const T *src, int64_t st, int row0,
                                           int nrows) {
    constexpr int LD = D + 4;
    constexpr int CPR = D / 4;
    for (int c = threadIdx.x; c < B * CPR; c += NT) {
        const int r = c / CPR, cc = c - r * CPR;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < nrows) x = load4(src + (int64_t)(row0 + r) * st + cc * 4);
        *reinterpret_cast<float4 *>(dst + r * LD + cc * 4) = x;
    }
}

// Per-row softmax statistics of a query block: lse in the base-2 domain
// (+inf for rows that do not exist or admit no key, so that P = 0 there) and Dr.
__device__ __forceinline__ void stage_row_stats(float *s_lse2, float *s_dr, const float *lse,
                                                const float *dr, int64_t row_base, int row0,
                                                int nrows) {
    for (int r = threadIdx.x; r < B; r += NT) {
        float l2 = INFINITY, d = 0.f;
        if (row0 + r < nrows) {
            const float x = lse[row_base + row0 + r];
            l2 = (x == -INFINITY) ? INFINITY : x * kLog2e;
            d = dr[row_base + row0 + r];
        }
        s_lse2[r] = l2;
        s_dr[r] = d;
    }
}

// Score-shaped micro-tile: acc[r][c] = <A[ty + 16 r], B[tx + 16 c]> over D.
template <int D>
__device__ __forceinline__ void tile_nt(float (&acc)[4][4], const float *A, const float *Bm,
                                        int tx, int ty) {
    constexpr int LD = D + 4;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
        float4 a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4 *>(A + (ty + 16 * r) * LD + d);
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = *reinterpret_cast<const float4 *>(Bm + (tx + 16 * c) * LD + d);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[r][c] = fmaf(a[r].x, b[c].x, acc[r][c]);
                acc[r][c] = fmaf(a[r].y, b[c].y, acc[r][c]);
                acc[r][c] = fmaf(a[r].z, b[c].z, acc[r][c]);
                acc[r][c] = fmaf(a[r].w, b[c].w, acc[r][c]);
            }
    }
}

// ---- preprocess: Dr = rowsum(dO * O), and lse in the base-2 domain ----------

constexpr int kRowDotRows = 4;  // rows per warp with loads in flight at once

// One warp per row r = t * H + h (token t, head h); each pass of a warp issues
// the loads of kRowDotRows rows before reducing any, so that enough bytes are
// in flight per SM to cover the HBM latency.  Rows are numbered in int64
// (n_q * H * 32 threads can exceed 2^32); a warp's rows are nwarps apart, so
// (t, h) advance by a fixed step without a division per row.
template <typename Tin, typename To, int D>
__global__ void __launch_bounds__(256) row_dot_kernel(const BwdParams p) {
    pdl_trigger();
    pdl_wait();
    static_assert(D <= 128, "one 4-column chunk per lane");
    constexpr int U = kRowDotRows;
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)p.n_q * p.H;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t r_first = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t step_t = nwarps / p.H;
    const int step_h = (int)(nwarps - step_t * p.H);
    int64_t t = r_first / p.H;
    int h = (int)(r_first - t * p.H);
    const int d = 4 * lane;  // lanes past D idle
    for (int64_t r0 = r_first; r0 < rows; r0 += U * nwarps) {
        // all loads of the pass (lse included) are issued before any store
        float4 a[U], b[U];
        float x[U];
        int64_t at[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool live = r0 + u * nwarps < rows;
            at[u] = (int64_t)h * p.n_q + t;
            a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            x[u] = 0.f;
            if (live && d < D) {
                a[u] = load4(static_cast<const Tin *>(p.dout) + t * p.do_st + (int64_t)h * p.do_sh + d);
                b[u] = load4(static_cast<const To *>(p.o) + t * p.o_st + (int64_t)h * p.o_sh + d);
            }
            if (live && lane == 0) x[u] = __ldg(p.lse + at[u]);
            t += step_t;
            h += step_h;
            if (h >= p.H) {
                h -= p.H;
                ++t;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float acc = a[u].x * b[u].x + a[u].y * b[u].y + a[u].z * b[u].z + a[u].w * b[u].w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && r0 + u * nwarps < rows) {
                p.dr[at[u]] = acc;
                p.lse2[at[u]] = x[u] == -INFINITY ? INFINITY : x[u] * kLog2e;
            }
        }
    }
}

// ---- dK, dV ----------------------------------------------------------------

template <int D>
constexpr size_t dkdv_smem_bytes() {
    return sizeof(float) * (size_t)(4 * B * (D + 4) + 2 * B * LDP + 2 * B);
}

template <typename Tin, typename Tg, int D>
__global__ void __launch_bounds__(NT) dkdv_simt_kernel(const BwdParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int LD = D + 4;
    constexpr int NG = D / 64;
    extern __shared__ float4 smem4[];
    float *sK = reinterpret_cast<float *>(smem4);
    float *sV = sK + B * LD;
    float *sQ = sV + B * LD;
    float *sdO = sQ + B * LD;
    float *sP = sdO + B * LD;
    float *sdS = sP + B * LDP;
    float *s_lse2 = sdS + B * LDP;
    float *s_dr = s_lse2 + B;
    __shared__ int s_w;

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int total = p.sched_kv.hdr[1];
    const Tin *gq = static_cast<const Tin *>(p.q);
    const Tin *gk = static_cast<const Tin *>(p.k);
    const Tin *gv = static_cast<const Tin *>(p.v);
    const Tin *gdo = static_cast<const Tin *>(p.dout);

    for (;;) {
        if (tid == 0) s_w = atomicAdd(p.sched_kv.hdr, 1);
        __syncthreads();
        const int w = s_w;
        __syncthreads();
        if (w >= total) break;
        // causal: earlier key blocks are seen by more query blocks, so run them first
        const WorkItem it = map_item(w, p.sched_kv.prefix, p.n_seq, p.H, false);
        int q_start, Lq, k_start, Lk;
        seq_bounds(p.cu_q, p.n_q, it.b, q_start, Lq);
        seq_bounds(p.cu_k, p.n_k, it.b, k_start, Lk);
        const int key0 = it.t * B, h = it.h;

        stage_tile<Tin, D>(sK, gk + (int64_t)k_start * p.k_st + (int64_t)h * p.k_sh, p.k_st, key0, Lk);
        stage_tile<Tin, D>(sV, gv + (int64_t)k_start * p.v_st + (int64_t)h * p.v_sh, p.v_st, key0, Lk);

        float dk[4][NG * 4], dv[4][NG * 4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < NG * 4; ++e) dk[r][e] = dv[r][e] = 0.f;

        const int qb_first = p.causal ? key0 / B : 0;
        const int qb_end = (Lq + B - 1) / B;
        const Tin *qbase = gq + (int64_t)q_start * p.q_st + (int64_t)h * p.q_sh;
        const Tin *dobase = gdo + (int64_t)q_start * p.do_st + (int64_t)h * p.do_sh;
        const int64_t stat_base = (int64_t)h * p.n_q + q_start;

        for (int qb = qb_first; qb < qb_end; ++qb) {
            const int row0 = qb * B;
            __syncthreads();
            stage_tile<Tin, D>(sQ, qbase, p.q_st, row0, Lq);
            stage_tile<Tin, D>(sdO, dobase, p.do_st, row0, Lq);
            stage_row_stats(s_lse2, s_dr, p.lse, p.dr, stat_base, row0, Lq);
            __syncthreads();

            float s[4][4], dp[4][4];
            tile_nt<D>(s, sQ, sK, tx, ty);
            tile_nt<D>(dp, sdO, sV, tx, ty);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int rl = ty + 16 * r, row = row0 + rl;
                const float l2 = s_lse2[rl], drr = s_dr[rl];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int key = key0 + tx + 16 * c;
                    const bool ok = key < Lk && (!p.causal || key <= row);
                    const float pr = ok ? exp2_approx(s[r][c] * p.scale_log2 - l2) : 0.f;
                    sP[rl * LDP + tx + 16 * c] = pr;
                    sdS[rl * LDP + tx + 16 * c] = pr * (dp[r][c] - drr);
                }
            }
            __syncthreads();

            // dV[key] += sum_row P[row][key] dO[row];  dK[key] += sum_row dS[row][key] Q[row]
#pragma unroll 2
            for (int row = 0; row < B; ++row) {
                float pk[4], sk[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    pk[r] = sP[row * LDP + ty + 16 * r];
                    sk[r] = sdS[row * LDP + ty + 16 * r];
                }
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float4 o4 = *reinterpret_cast<const float4 *>(sdO + row * LD + 64 * g + 4 * tx);
                    const float4 q4 = *reinterpret_cast<const float4 *>(sQ + row * LD + 64 * g + 4 * tx);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        dv[r][4 * g + 0] = fmaf(pk[r], o4.x, dv[r][4 * g + 0]);
                        dv[r][4 * g + 1] = fmaf(pk[r], o4.y, dv[r][4 * g + 1]);
                        dv[r][4 * g + 2] = fmaf(pk[r], o4.z, dv[r][4 * g + 2]);
                        dv[r][4 * g + 3] = fmaf(pk[r], o4.w, dv[r][4 * g + 3]);
                        dk[r][4 * g + 0] = fmaf(sk[r], q4.x, dk[r][4 * g + 0]);
                        dk[r][4 * g + 1] = fmaf(sk[r], q4.y, dk[r][4 * g + 1]);
                        dk[r][4 * g + 2] = fmaf(sk[r], q4.z, dk[r][4 * g + 2]);
                        dk[r][4 * g + 3] = fmaf(sk[r], q4.w, dk[r][4 * g + 3]);
                    }
                }
            }
        }

        Tg *gdk = static_cast<Tg *>(p.dk);
        Tg *gdv = static_cast<Tg *>(p.dv);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int key = key0 + ty + 16 * r;
            if (key >= Lk) continue;
            Tg *dkrow = gdk + (int64_t)(k_start + key) * p.dk_st + (int64_t)h * p.dk_sh;
            Tg *dvrow = gdv + (int64_t)(k_start + key) * p.dv_st + (int64_t)h * p.dv_sh;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                store4(dkrow + 64 * g + 4 * tx,
                       make_float4(dk[r][4 * g] * p.scale, dk[r][4 * g + 1] * p.scale,
                                   dk[r][4 * g + 2] * p.scale, dk[r][4 * g + 3] * p.scale));
                store4(dvrow + 64 * g + 4 * tx,
                       make_float4(dv[r][4 * g], dv[r][4 * g + 1], dv[r][4 * g + 2], dv[r][4 * g + 3]));
            }
        }
    }
}

// ---- dQ --------------------------------------------------------------------

template <int D>
constexpr size_t dq_smem_bytes() {
    return sizeof(float) * (size_t)(4 * B * (D + 4) + B * LDP + 2 * B);
}

template <typename Tin, typename Tg, int D>
__global__ void __launch_bounds__(NT) dq_simt_kernel(const BwdParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int LD = D + 4;
    constexpr int NG = D / 64;
    extern __shared__ float4 smem4[];
    float *sQ = reinterpret_cast<float *>(smem4);
    float *sdO = sQ + B * LD;
    float *sK = sdO + B * LD;
    float *sV = sK + B * LD;
    float *sdS = sV + B * LD;
    float *s_lse2 = sdS + B * LDP;
    float *s_dr = s_lse2 + B;
    __shared__ int s_w;

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int total = p.sched_q.hdr[1];
    const Tin *gq = static_cast<const Tin *>(p.q);
    const Tin *gk = static_cast<const Tin *>(p.k);
    const Tin *gv = static_cast<const Tin *>(p.v);
    const Tin *gdo = static_cast<const Tin *>(p.dout);

    for (;;) {
        if (tid == 0) s_w = atomicAdd(p.sched_q.hdr, 1);
        __syncthreads();
        const int w = s_w;
        __syncthreads();
        if (w >= total) break;
        const WorkItem it = map_item(w, p.sched_q.prefix, p.n_seq, p.H, true);
        int q_start, Lq, k_start, Lk;
        seq_bounds(p.cu_q, p.n_q, it.b, q_start, Lq);
        seq_bounds(p.cu_k, p.n_k, it.b, k_start, Lk);
        const int row0 = it.t * B, h = it.h;

        stage_tile<Tin, D>(sQ, gq + (int64_t)q_start * p.q_st + (int64_t)h * p.q_sh, p.q_st, row0, Lq);
        stage_tile<Tin, D>(sdO, gdo + (int64_t)q_start * p.do_st + (int64_t)h * p.do_sh, p.do_st, row0, Lq);
        stage_row_stats(s_lse2, s_dr, p.lse, p.dr, (int64_t)h * p.n_q + q_start, row0, Lq);

        float dq[4][NG * 4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < NG * 4; ++e) dq[r][e] = 0.f;

        const int n_keys = p.causal ? min(Lk, row0 + B) : Lk;
        const int n_tiles = (n_keys + B - 1) / B;
        const Tin *kbase = gk + (int64_t)k_start * p.k_st + (int64_t)h * p.k_sh;
        const Tin *vbase = gv + (int64_t)k_start * p.v_st + (int64_t)h * p.v_sh;

        for (int kt = 0; kt < n_tiles; ++kt) {
            const int key0 = kt * B;
            __syncthreads();
            stage_tile<Tin, D>(sK, kbase, p.k_st, key0, Lk);
            stage_tile<Tin, D>(sV, vbase, p.v_st, key0, Lk);
            __syncthreads();

            float s[4][4], dp[4][4];
            tile_nt<D>(s, sQ, sK, tx, ty);
            tile_nt<D>(dp, sdO, sV, tx, ty);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int rl = ty + 16 * r, row = row0 + rl;
                const float l2 = s_lse2[rl], drr = s_dr[rl];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int key = key0 + tx + 16 * c;
                    const bool ok = key < Lk && (!p.causal || key <= row);
                    const float pr = ok ? exp2_approx(s[r][c] * p.scale_log2 - l2) : 0.f;
                    sdS[rl * LDP + tx + 16 * c] = pr * (dp[r][c] - drr);
                }
            }
            __syncthreads();

            // dQ[row] += sum_key dS[row][key] K[key]
#pragma unroll 2
            for (int j = 0; j < B; j += 4) {
                float4 sr[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) sr[r] = *reinterpret_cast<const float4 *>(sdS + (ty + 16 * r) * LDP + j);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const float4 kk = *reinterpret_cast<const float4 *>(sK + (j + jj) * LD + 64 * g + 4 * tx);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float sj = jj == 0 ? sr[r].x : jj == 1 ? sr[r].y : jj == 2 ? sr[r].z : sr[r].w;
                            dq[r][4 * g + 0] = fmaf(sj, kk.x, dq[r][4 * g + 0]);
                            dq[r][4 * g + 1] = fmaf(sj, kk.y, dq[r][4 * g + 1]);
                            dq[r][4 * g + 2] = fmaf(sj, kk.z, dq[r][4 * g + 2]);
                            dq[r][4 * g + 3] = fmaf(sj, kk.w, dq[r][4 * g + 3]);
                        }
                    }
                }
            }
        }

        Tg *gdq = static_cast<Tg *>(p.dq);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = row0 + ty + 16 * r;
            if (row >= Lq) continue;
            Tg *dqrow = gdq + (int64_t)(q_start + row) * p.dq_st + (int64_t)h * p.dq_sh;
#pragma unroll
            for (int g = 0; g < NG; ++g)
                store4(dqrow + 64 * g + 4 * tx,
                       make_float4(dq[r][4 * g] * p.scale, dq[r][4 * g + 1] * p.scale,
                                   dq[r][4 * g + 2] * p.scale, dq[r][4 * g + 3] * p.scale));
        }
    }
}

// ---- launchers -------------------------------------------------------------

template <typename K>
cudaError_t launch_persistent(K kern, size_t smem, int num_ctas, const BwdParams &p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (num_ctas <= 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
        if (e != cudaSuccess) return e;
        num_ctas = sm_count() * (per_sm > 0 ? per_sm : 1);
    }
    e = launch_pdl(kern, dim3(num_ctas), dim3(NT), smem, s, p);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tin, typename Tg, int D>
cudaError_t bwd_typed(const BwdParams &p, int num_ctas, cudaStream_t s, bool dkdv) {
    if (dkdv) return launch_persistent(dkdv_simt_kernel<Tin, Tg, D>, dkdv_smem_bytes<D>(), num_ctas, p, s);
    return launch_persistent(dq_simt_kernel<Tin, Tg, D>, dq_smem_bytes<D>(), num_ctas, p, s);
}

template <typename Tin, int D>
cudaError_t bwd_grad(const BwdParams &p, int num_ctas, cudaStream_t s, bool dkdv) {
    if (p.grad_dtype == ATTN_F32) return bwd_typed<Tin, float, D>(p, num_ctas, s, dkdv);
    return bwd_typed<Tin, Tin, D>(p, num_ctas, s, dkdv);
}

template <int D>
cudaError_t bwd_d(const BwdParams &p, int num_ctas, cudaStream_t s, bool dkdv) {
    switch (p.dtype) {
    case ATTN_F16: return bwd_grad<__half, D>(p, num_ctas, s, dkdv);
    case ATTN_BF16: return bwd_grad<__nv_bfloat16, D>(p, num_ctas, s, dkdv);
    default: return bwd_typed<float, float, D>(p, num_ctas, s, dkdv);
    }
}

template <typename Tin, typename To, int D>
cudaError_t row_dot_typed(const BwdParams &p, cudaStream_t s) {
    const int64_t rows = (int64_t)p.n_q * p.H;
    if (rows == 0) return cudaSuccess;
    // 8 warps per block, kRowDotRows rows per warp and pass; at most one wave of
    // resident blocks (a second wave would leave the first one's SMs idle at its tail)
    static int per_sm = 0;  // resident blocks per SM of this instantiation
    if (per_sm == 0 &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_dot_kernel<Tin, To, D>, 256, 0) != cudaSuccess)
        per_sm = 1;
    const int64_t want = (rows + 8 * kRowDotRows - 1) / (8 * kRowDotRows);
    const int64_t cap = (int64_t)(per_sm > 0 ? per_sm : 1) * sm_count();
    const cudaError_t e = launch_pdl(row_dot_kernel<Tin, To, D>, dim3((int)(want < cap ? want : cap)), dim3(256), 0, s, p);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tin, int D>
cudaError_t row_dot_o(const BwdParams &p, cudaStream_t s) {
    if (p.o_dtype == ATTN_F32) return row_dot_typed<Tin, float, D>(p, s);
    return row_dot_typed<Tin, Tin, D>(p, s);
}

template <int D>
cudaError_t row_dot_d(const BwdParams &p, cudaStream_t s) {
    switch (p.dtype) {
    case ATTN_F16: return row_dot_o<__half, D>(p, s);
    case ATTN_BF16: return row_dot_o<__nv_bfloat16, D>(p, s);
    default: return row_dot_typed<float, float, D>(p, s);
    }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams &p, cudaStream_t s) {
    if ((int64_t)p.n_q * p.H == 0) return cudaSuccess;
    return p.D == 64 ? row_dot_d<64>(p, s) : row_dot_d<128>(p, s);
}

cudaError_t launch_bwd_dkdv_simt(const BwdParams &p, int num_ctas, cudaStream_t s) {
    return p.D == 64 ? bwd_d<64>(p, num_ctas, s, true) : bwd_d<128>(p, num_ctas, s, true);
}

cudaError_t launch_bwd_dq_simt(const BwdParams &p, int num_ctas, cudaStream_t s) {
    return p.D == 64 ? bwd_d<64>(p, num_ctas, s, false) : bwd_d<128>(p, num_ctas, s, false);
}

}  // namespace attn

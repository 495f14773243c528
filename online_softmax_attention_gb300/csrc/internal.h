// Internal (not exported) parameter blocks and launchers of the attention
// library.  The C ABI in attn_api.cu validates the public argument structs and
// translates them into these plain-old-data blocks, which kernels take by value.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

// Schedule block in the workspace: [0] dynamic work counter, [1] item count,
// then the per-sequence prefix of item counts (n_seq + 1 ints).
constexpr int kSchedHeaderInts = 16;

struct Sched {
    int *hdr;          // counter, total
    const int *prefix; // n_seq + 1 entries
};

struct FwdParams {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh, o_st, o_sh;
    int n_q, n_k, H, D;
    float scale;       // score scale
    float scale_log2;  // scale * log2(e)
    int causal;
    int dtype, o_dtype;
    int qk_fp8;        // q and k are e4m3 (one byte per element); v is `dtype`
    int n_seq;
    const int32_t *cu_q, *cu_k;  // null => one sequence
    Sched sched;
    // > 0: static schedule of one sequence (cu_q, cu_k null) with this many
    // work items, one per CTA of a grid of exactly this size; the workspace's
    // schedule block is neither written nor read.  0: dynamic schedule.
    int static_items;
    int *status;
    long long watchdog_cycles;
    // split-K: key tiles of every query tile cut into n_splits chunks; chunk c
    // writes its partial (O_c f32, lse_c) at o + c * o_split_st, lse + c * lse_split_st
    int n_splits;
    int64_t o_split_st, lse_split_st;
    // tile pruning: prune a key tile when its largest score (log2 units) is
    // below the query tile's rolling max + prune_log2; count pruned tiles
    int prune;
    float prune_log2;  // log2(rho)
    unsigned long long *pruned_tiles;
    // f32 inputs on the tensor cores: workspace region for the bf16 parts of
    // q, k and v (see fwd_x3.cu), else null
    void *split_ws;
};

// Key-tile range [begin, end) of chunk c when n_tiles key tiles are cut into
// n_splits contiguous chunks of ceil(n_tiles / n_splits) tiles (the last ones
// may be shorter or empty).
struct KeyChunk {
    int begin, end;
};
#ifdef __CUDACC__
__host__ __device__
#endif
inline KeyChunk key_chunk(int n_tiles, int n_splits, int c) {
    const int per = (n_tiles + n_splits - 1) / n_splits;
    int b = c * per, e = b + per;
    if (b > n_tiles) b = n_tiles;
    if (e > n_tiles) e = n_tiles;
    return KeyChunk{b, e};
}

struct MergeParams {
    const float *o_parts, *lse_parts;
    void *o;
    float *lse;
    int64_t o_st, o_sh;        // output strides (elements)
    int64_t part_st;           // elements between partials of o_parts (n_q * H * D)
    int n_parts, n_q, H, D, o_dtype;
};

// Attention over a CSR relation (row_ptr over destination rows, col = sources).
struct CsrParams {
    const int64_t *row_ptr;
    const int32_t *col;
    int64_t n_edges;
    int n_dst, n_src, H, D;
    const float *scores;  // (n_edges, H) field scores, or null: dot-product scores
    const void *q, *k, *v;
    void *o;
    float *lse;
    int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh, o_st, o_sh;
    float scale_log2;
    int dtype, o_dtype;
    const int32_t *row_order;  // n_dst rows in processing order, or null: identity
    int *status;
};

cudaError_t launch_csr_fwd(const CsrParams &p, cudaStream_t s);

struct BwdParams {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh, o_st, o_sh, do_st, do_sh;
    int64_t dq_st, dq_sh, dk_st, dk_sh, dv_st, dv_sh;
    int n_q, n_k, H, D;
    float scale, scale_log2;
    int causal;
    int dtype, o_dtype, grad_dtype;
    int n_seq;
    const int32_t *cu_q, *cu_k;
    float *dr;          // (H, n_q) rowsum(dO * O), in the workspace
    float *lse2;        // (H, n_q) lse * log2(e), +inf where lse = -inf, in the workspace
    // fused dQ (tensor-core dK/dV kernel also accumulates dQ): f32 partial sums
    // laid out (H, D/4, n_q, 4) in the workspace, so that 32 consecutive query
    // rows of one 4-column group are 512 contiguous bytes; null = separate dQ kernel
    float *dq_accum;
    Sched sched_kv;     // items over key blocks (dk, dv)
    Sched sched_q;      // items over query blocks (dq)
    int *status;
    long long watchdog_cycles;
};

// Schedule preparation: validates cu_seqlens on the device and writes the
// prefix of item counts for tiles of `block` rows of the `cu_rows` side.
// Each tile counts as `splits` work items (split-K), numbered tile-major.
cudaError_t launch_prep(const int32_t *cu_q, const int32_t *cu_k, int n_seq, int n_q, int n_k,
                        int H, int block, int causal, int rows_are_keys, int splits, Sched sched,
                        int *status, cudaStream_t s);

// Merge of partial results (split-K): one warp per (query row, head).
cudaError_t launch_merge(const MergeParams &p, cudaStream_t s);

// SIMT (CUDA-core) kernels: any dtype, D in {64, 128}.
constexpr int kSimtBlock = 64;
cudaError_t launch_fwd_simt(const FwdParams &p, int num_ctas, cudaStream_t s);
int fwd_simt_ctas_per_sm(const FwdParams &p);  // resident CTAs per SM of the kernel p selects
cudaError_t launch_bwd_preprocess(const BwdParams &p, cudaStream_t s);
cudaError_t launch_bwd_dkdv_simt(const BwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dq_simt(const BwdParams &p, int num_ctas, cudaStream_t s);
// fused dQ: zero the partial sums (before the dK/dV kernel); dq = scale * sums
// converted to grad_dtype with dq's strides (after it)
cudaError_t launch_dq_accum_zero(const BwdParams &p, cudaStream_t s);
cudaError_t launch_dq_accum_convert(const BwdParams &p, cudaStream_t s);

// Number of multiprocessors of the current device.
int sm_count();

#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may start while the
// kernel before it on the stream is still running (once every CTA of that one
// has started and executed pdl_trigger).  Every kernel launched this way
// executes pdl_wait -- which returns once the previous grid has completed and
// its writes are visible -- before it reads global memory, so it sees that
// kernel's results; what it overlaps is its launch and set-up.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}
#endif

// Kernel-launch accounting (attn_launch_count).
void count_launch(int n = 1);

}  // namespace attn

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
    int n_seq;
    const int32_t *cu_q, *cu_k;  // null => one sequence
    Sched sched;
    int *status;
    long long watchdog_cycles;
};

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
    Sched sched_kv;     // items over key blocks (dk, dv)
    Sched sched_q;      // items over query blocks (dq)
    int *status;
    long long watchdog_cycles;
};

// Schedule preparation: validates cu_seqlens on the device and writes the
// prefix of item counts for tiles of `block` rows of the `cu_rows` side.
cudaError_t launch_prep(const int32_t *cu_q, const int32_t *cu_k, int n_seq, int n_q, int n_k,
                        int H, int block, int causal, int rows_are_keys, Sched sched,
                        int *status, cudaStream_t s);

// SIMT (CUDA-core) kernels: any dtype, D in {64, 128}.
constexpr int kSimtBlock = 64;
cudaError_t launch_fwd_simt(const FwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdParams &p, cudaStream_t s);
cudaError_t launch_bwd_dkdv_simt(const BwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dq_simt(const BwdParams &p, int num_ctas, cudaStream_t s);

// Number of multiprocessors of the current device.
int sm_count();

// Kernel-launch accounting (attn_launch_count).
void count_launch(int n = 1);

}  // namespace attn

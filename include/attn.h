/*
 * attn.h -- C ABI of the GB300 (sm_103a) online-softmax attention library.
 *
 * Exact scaled dot-product attention, forward and fused backward, computed by
 * the online-softmax block recurrence on one GPU.
 *
 * Definition (TIGA-lang, "注意力与稠密关系" attention examples page, section
 * "全量注意力，无掩码", display equation):
 *     s_hij  = <k_hj, q_hi> * scale
 *     out_hi = sum_j softmax_j(s_hi.) v_hj
 * over a relation that decides which (i, j) pairs exist:
 *   ATTN_FULL    every key of the query's sequence (dense relation);
 *   ATTN_CAUSAL  keys j <= i of the query's sequence (same page, section
 *                "因果稠密关系", triangular relation).
 * With cu_seqlens the tokens form independent sequences back to back and no
 * pair crosses a sequence boundary (same page, section
 * "用图组合表达 varlen 因果注意力": block-diagonal relation, flash-attn's
 * cu_seqlens convention [0, L1, L1+L2, ...]).
 *
 * Algorithm (OCANNL "Module Ir.Online_softmax", fourth bullet): for each
 * query tile a scan over key blocks carries the running row max m and the
 * rescaled row sum l, accumulates the numerator U = sum p*v, and the last
 * block writes O = U / l.  A key block that runs past the end of a sequence
 * is a guarded tail padded with -inf scores.  The row log-sum-exp
 * lse = m + ln l (natural log, of the scaled scores) is written for the
 * backward.
 *
 * Backward (same page, third bullet): Dr_i = sum_d dO_id * O_id per row;
 * per pair recompute p and dp = <dO_i, v_j>; ds = p * (dp - Dr_i);
 * dq = scale * ds . k, dk = scale * ds^T . q, dv = p^T . dO.  In the page's
 * layout each gradient has a nest of its own that owns what it writes
 * (ATTN_DQ_SEPARATE: no atomics, run-to-run deterministic); ATTN_DQ_FUSED
 * instead folds the dq nest into the dk/dv nest with f32 reductions (see
 * attn_dq_mode).
 *
 * Conventions for every entry point:
 *  - Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *    owned by the caller.  The library allocates no memory visible to the
 *    caller; scratch comes from the caller's workspace.
 *  - Tensors are (tokens, heads, D) with element strides given per tensor for
 *    the token and head axes; the D axis must be contiguous (stride 1).
 *    Token and head strides must be multiples of 8 elements for 16-bit types
 *    and of 4 elements for f32 (16-byte rows), and base pointers must be
 *    16-byte aligned.
 *  - lse / Dr are f32 (H, n_q) contiguous.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  No call synchronises the host, except
 *    attn_device_status().
 *  - Return value: ATTN_OK (0) or a negative attn_status.  Invalid arguments
 *    are rejected before any launch.  Errors found by kernels (inconsistent
 *    cu_seqlens, a watchdog timeout) are reported by attn_device_status().
 *  - Outputs are fully overwritten; no zero-initialisation is needed.
 *  - A query row that admits no key (only an empty key sequence under
 *    ATTN_FULL) gets O = 0 and lse = -inf.
 *  - Inputs must be finite.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 6

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_EINVAL = -1,        /* bad pointer, stride, size or cu_seqlens */
    ATTN_EUNSUPPORTED = -2,  /* valid but not implemented (dtype, D, relation mix, GPU) */
    ATTN_ECUDA = -3,         /* a CUDA runtime call failed; see attn_last_error_string() */
    ATTN_ETIMEOUT = -4,      /* a kernel's bounded wait expired (device watchdog) */
    ATTN_EWORKSPACE = -5     /* workspace missing or smaller than *_workspace_bytes() */
} attn_status;

typedef enum attn_dtype { ATTN_F16 = 0, ATTN_BF16 = 1, ATTN_F32 = 2 } attn_dtype;

typedef enum attn_relation { ATTN_FULL = 0, ATTN_CAUSAL = 1 } attn_relation;

/* Kernel choice.  AUTO picks the tcgen05 tensor-core kernels for f16/bf16 and
 * the FP32 SIMT kernels for f32.  SIMT forces the CUDA-core kernels (any
 * dtype); TC forces the tensor-core kernels (f16/bf16 only). */
typedef enum attn_kernel { ATTN_KERNEL_AUTO = 0, ATTN_KERNEL_SIMT = 1, ATTN_KERNEL_TC = 2 } attn_kernel;

/* How the backward computes dq.
 * SEPARATE: dk/dv by one kernel (per key block, loop over query blocks) and
 *   dq by another (per query block, loop over key blocks), each writing its
 *   gradient once: deterministic, but the dq kernel recomputes the scores and
 *   dp of every pair (7 contractions per pair in all).
 * FUSED: the dk/dv kernel also forms dq's per-pair contribution ds . k
 *   (5 contractions per pair) and adds it with f32 reductions to partial sums
 *   in the workspace; the dq stage scales and converts the sums.  The order of
 *   the additions varies from run to run, so dq may differ in the last bits
 *   between runs.  Tensor-core kernels only (ATTN_EUNSUPPORTED with SIMT).
 * AUTO: SEPARATE (on the causal training shapes the fused kernel's f32
 *   reduction traffic, 64 KiB per pair of 128-row tiles, costs more than the
 *   recomputation it saves). */
typedef enum attn_dq_mode { ATTN_DQ_AUTO = 0, ATTN_DQ_SEPARATE = 1, ATTN_DQ_FUSED = 2 } attn_dq_mode;

/* A (tokens, heads, D) tensor view: element strides of the token and head axes. */
typedef struct attn_tensor {
    void *ptr;
    int64_t stride_tok;
    int64_t stride_head;
} attn_tensor;

typedef struct attn_fwd_args {
    attn_tensor q;        /* in:  (n_q, H, D), dtype */
    attn_tensor k;        /* in:  (n_k, H, D), dtype */
    attn_tensor v;        /* in:  (n_k, H, D), dtype */
    attn_tensor o;        /* out: (n_q, H, D), o_dtype */
    float *lse;           /* out: (H, n_q) f32, natural-log row log-sum-exp; may be NULL */
    int32_t n_q, n_k;     /* total query / key tokens */
    int32_t H, D;         /* heads; head dim (64 or 128) */
    float scale;          /* score scale, usually D^-1/2: any finite value (0 gives the
                             uniform average of the admitted values, a negative one
                             is accepted); NaN or +-inf: ATTN_EINVAL */
    int32_t relation;     /* attn_relation */
    int32_t dtype;        /* attn_dtype of q, k, v */
    int32_t o_dtype;      /* attn_dtype of o: dtype or ATTN_F32 */
    int32_t n_seq;        /* sequences; 1 when cu_seqlens_* are NULL */
    const int32_t *cu_seqlens_q; /* device, n_seq+1 offsets from 0, or NULL (one sequence of n_q) */
    const int32_t *cu_seqlens_k; /* device, n_seq+1 offsets from 0, or NULL (one sequence of n_k) */
    void *workspace;      /* device scratch, attn_fwd_workspace_bytes() bytes, 256-byte aligned */
    size_t workspace_bytes;
    int32_t kernel;       /* attn_kernel */
    int32_t num_ctas;     /* persistent grid size; 0 = one per SM */
    int32_t num_splits;   /* key splits per query tile (split-K): 0 = chosen by the
                             library (see attn_fwd_num_splits), 1 = none, 2..ATTN_MAX_SPLITS */
    float prune_threshold; /* tile pruning (approximate forward, see below): 0 = off,
                              the exact forward; 0 < rho <= 1 enables it */
    uint64_t *pruned_tiles; /* optional device counter, or NULL: with pruning on, the
                               forward adds the number of pruned tiles to it */
    int32_t qk_fp8;       /* 0: q and k are `dtype`; 1: q and k are fp8 e4m3 (see below) */
} attn_fwd_args;

/* fp8 queries and keys (qk_fp8 = 1; no counterpart on the pages, a use of the
 * sm_103a tensor cores' 8-bit score contraction): q and k hold e4m3 values,
 * one byte per element (strides in elements = bytes, rows 16-byte aligned);
 * v is `dtype` (f16 or bf16), P is rounded to it and o is o_dtype as usual.
 * The scores are the exact products of the e4m3 values accumulated in f32,
 * times `scale`; a caller with per-tensor dequantisation factors for q and k
 * folds them into `scale`.  Tensor-core kernel only: D = 128 and scale > 0,
 * else ATTN_EUNSUPPORTED (also with ATTN_KERNEL_SIMT).  Backward: none. */

/* Tile pruning (TIGA-lang attention examples page, section
 * "基于 tile 剪枝的稀疏注意力", tile-pruned sparse attention): an explicit,
 * approximate option of the forward.  A tile pairs a query tile with a key
 * tile of the kernel's own sizes (128 x 128 for the tensor-core kernel, 64 x 64
 * for the SIMT kernel).  Per query tile the key tiles are scanned in order;
 * every tile's scores are computed, and a tile whose largest score m_tile
 * satisfies  m_tile < m_run + ln(rho)  -- m_run being the largest score of the
 * tiles admitted so far for that query tile -- is pruned: it adds nothing to
 * the softmax or to O (its value tile is still loaded).  The rule bounds no
 * per-row error.  Only the full relation over one sequence (no cu_seqlens) and
 * no key splits are supported; other combinations, and any backward call with
 * a non-zero prune_threshold, return ATTN_EUNSUPPORTED (fail closed). */

/* Upper bound of attn_fwd_args.num_splits and of attn_merge_args.n_parts. */
#define ATTN_MAX_SPLITS 64

typedef struct attn_bwd_args {
    attn_tensor q, k, v;  /* in: as in the forward */
    attn_tensor o;        /* in: forward output, o_dtype */
    attn_tensor dout;     /* in: dL/dO, (n_q, H, D), dtype */
    const float *lse;     /* in: (H, n_q) f32 from attn_fwd */
    attn_tensor dq;       /* out: (n_q, H, D), grad_dtype */
    attn_tensor dk;       /* out: (n_k, H, D), grad_dtype */
    attn_tensor dv;       /* out: (n_k, H, D), grad_dtype */
    int32_t n_q, n_k, H, D;
    float scale;
    int32_t relation, dtype, o_dtype;
    int32_t grad_dtype;   /* attn_dtype of dq, dk, dv: dtype or ATTN_F32 */
    int32_t n_seq;
    const int32_t *cu_seqlens_q, *cu_seqlens_k;
    void *workspace;      /* attn_bwd_workspace_bytes() bytes, 256-byte aligned */
    size_t workspace_bytes;
    int32_t kernel;
    int32_t num_ctas;
    float prune_threshold; /* must be 0: the backward of a tile-pruned forward is not
                              defined, and a non-zero value returns ATTN_EUNSUPPORTED */
    int32_t dq_mode;      /* attn_dq_mode */
} attn_bwd_args;

/* Partial attention results over disjoint key sets, to be merged
 * (attn_merge).  Partial c is attention of the same query rows over its own
 * key set: its output O_c (normalised by its own row sum) and its row
 * log-sum-exp lse_c (-inf when it admits no key; O_c is then ignored). */
typedef struct attn_merge_args {
    const float *o_parts;   /* in:  (n_parts, n_q, H, D) f32, contiguous */
    const float *lse_parts; /* in:  (n_parts, H, n_q) f32, contiguous */
    attn_tensor o;          /* out: (n_q, H, D), o_dtype; may not overlap the inputs */
    float *lse;             /* out: (H, n_q) f32, or NULL */
    int32_t n_parts;        /* 1..ATTN_MAX_SPLITS */
    int32_t n_q, H, D;      /* D: a multiple of 4, at most 256 */
    int32_t o_dtype;        /* attn_dtype */
} attn_merge_args;

/* Attention over a general CSR relation (TIGA-lang attention examples page:
 * the varlen section writes a relation as an explicit CSR graph of exactly
 * the admitted edges; the GAT section's display equation is a softmax over
 * each row's incoming edges):
 *     out[i, h] = sum_{e in row i} exp(s[e, h]) / sum_{e' in row i} exp(s[e', h]) * v[col[e], h]
 * Row i's edges are col_idx[row_ptr[i] .. row_ptr[i+1]); an edge listed twice
 * counts twice.  The score is the field edge_scores[e, h] (segment softmax)
 * or, with edge_scores NULL, scale * <q[i, h], k[col[e], h]>.  A row without
 * edges gets O = 0, lse = -inf.  Malformed relations (offsets that decrease
 * or leave [0, n_edges], sources outside [0, n_src)) are not read out of
 * bounds: the row or edge is skipped and attn_device_status() reports
 * ATTN_EINVAL.  One kernel on `stream`; no workspace. */
typedef struct attn_csr_args {
    const int64_t *row_ptr;   /* device, n_dst + 1 nondecreasing offsets in [0, n_edges] */
    const int32_t *col_idx;   /* device, n_edges source indices */
    int64_t n_edges;
    int32_t n_dst, n_src;     /* destination rows; source rows */
    int32_t H, D;             /* heads; D a multiple of 4, at most 256 */
    const float *edge_scores; /* device (n_edges, H) f32 field scores, or NULL */
    attn_tensor q;            /* (n_dst, H, D) dtype, dot-product scores only */
    attn_tensor k;            /* (n_src, H, D) dtype, dot-product scores only */
    attn_tensor v;            /* (n_src, H, D) dtype */
    attn_tensor o;            /* out: (n_dst, H, D) o_dtype */
    float *lse;               /* out: (H, n_dst) f32, or NULL */
    float scale;              /* dot-product scores only */
    int32_t dtype;            /* attn_dtype of q, k, v */
    int32_t o_dtype;          /* dtype or ATTN_F32 */
    /* device, n_dst entries: the order in which the kernel takes the rows (a
     * permutation of [0, n_dst)), or NULL for 0, 1, 2, ...  Results do not
     * depend on it, bit for bit; it only decides which rows are in flight
     * together, and so how often their sources' rows are found in the L2:
     * an order that keeps rows with shared sources close (e.g. points sorted
     * along a space-filling curve) turns most gathers into L2 hits.  An entry
     * outside [0, n_dst) is skipped and reported as ATTN_EINVAL; a row the
     * order omits is not written. */
    const int32_t *row_order;
} attn_csr_args;

/* Library ABI version (ATTN_ABI_VERSION) and struct sizes, for bindings to
 * check their mirrors of the structs above. */
ATTN_API int attn_abi_version(void);
ATTN_API size_t attn_fwd_args_size(void);
ATTN_API size_t attn_bwd_args_size(void);
ATTN_API size_t attn_merge_args_size(void);
ATTN_API size_t attn_csr_args_size(void);

/* Bytes of device workspace the call needs (depends on n_seq, H, n_q, and
 * for the forward on the number of key splits: n_splits > 1 adds the partial
 * results, n_splits * n_q * H * (D + 1) * 4 bytes; for the backward on the dq
 * mode: ATTN_DQ_FUSED adds the dq partial sums, n_q * H * D * 4 bytes).
 * Only sizes, dtypes, the relation, the kernel choice, num_splits and whether
 * cu_seqlens are given are read: the tensor and workspace pointers may still
 * be unset.  Arguments the call would reject give the unsplit size. */
ATTN_API size_t attn_fwd_workspace_bytes(const attn_fwd_args *a);
ATTN_API size_t attn_bwd_workspace_bytes(const attn_bwd_args *a);

/* Forward: writes o and lse.  Launches a schedule-preparation kernel and one
 * persistent attention kernel on `stream`; with key splits (split-K) the
 * attention kernel writes one partial result per split into the workspace
 * and a merge kernel (as attn_merge) combines them into o and lse.  One
 * sequence (no cu_seqlens) whose work items fit in one wave of the default
 * grid (num_ctas = 0) needs no preparation: the attention kernel then runs
 * one item per CTA and is the only launch (plus the merge when split). */
ATTN_API int attn_fwd(const attn_fwd_args *a, void *stream);

/* Key splits a forward with these arguments runs (>= 1), resolving
 * num_splits = 0, or a negative attn_status.  Host-only; launches nothing.
 *
 * Split-K (Vx issue "Chunked-dot Reduce lowering: shorten the reduction
 * dependency chain", measurement section: the record FP32 kernel splits the
 * keys in C = 8 chunks): each query tile's key tiles are cut into n_splits
 * contiguous chunks that run as separate work items, so shapes with few
 * query tiles still fill the GPU.  The automatic choice splits only when the
 * query tiles alone leave most SMs idle and every chunk keeps at least two
 * key tiles. */
ATTN_API int attn_fwd_num_splits(const attn_fwd_args *a);

/* Merge of partial results over disjoint key sets into attention over their
 * union (the split-K merge; with each partial's online-softmax state written
 * as m_c = lse_c, l_c = 1, U_c = O_c, this is the (m, l, U) combination of the
 * OCANNL "Module Ir.Online_softmax" page, fourth bullet):
 *     lse = ln sum_c exp(lse_c),   O = sum_c exp(lse_c - lse) O_c.
 * A row whose partials are all -inf gets O = 0, lse = -inf.  One kernel on
 * `stream`; no workspace. */
ATTN_API int attn_merge(const attn_merge_args *a, void *stream);

/* Backward: writes dq, dk, dv.  Equivalent to attn_bwd_preprocess, then
 * attn_bwd_dkdv, then attn_bwd_dq on the same stream and workspace. */
ATTN_API int attn_bwd(const attn_bwd_args *a, void *stream);

/* The three stages of attn_bwd, callable one by one (e.g. to time each):
 *  preprocess: Dr = rowsum(dO * O) into the workspace, and the schedules
 *              (FUSED: also zeroes the dq partial sums);
 *  dkdv:       per key block, loop over query blocks, write dk and dv
 *              (FUSED: also add each pair's dq contribution to the sums);
 *  dq:         SEPARATE: per query block, loop over key blocks, write dq;
 *              FUSED: dq = scale * partial sums, converted to grad_dtype.
 * dkdv and dq read what preprocess wrote into the same workspace. */
ATTN_API int attn_bwd_preprocess(const attn_bwd_args *a, void *stream);
ATTN_API int attn_bwd_dkdv(const attn_bwd_args *a, void *stream);
ATTN_API int attn_bwd_dq(const attn_bwd_args *a, void *stream);

/* Flat form for contiguous (N, H, D) self-attention tensors (token stride
 * H*D, head stride D), o in the input dtype, AUTO kernel choice and AUTO key
 * splits (the same schedule attn_fwd picks for these arguments).
 * cu_seqlens: device, n_seq+1 entries, or NULL for one sequence (n_seq is
 * then ignored).  workspace: device, 256-byte aligned, at least
 * attn_fwd_simple_workspace_bytes(N, H, D, relation, n_seq, dtype) bytes
 * (ATTN_EWORKSPACE otherwise).  Defined as in attn_fwd (TIGA-lang attention
 * examples page, section "全量注意力，无掩码", and its causal and varlen
 * sections). */
ATTN_API int attn_fwd_simple(const void *q, const void *k, const void *v, void *out, float *lse,
                    int32_t N, int32_t H, int32_t D, float scale, int32_t relation,
                    const int32_t *cu_seqlens, int32_t n_seq, int32_t dtype,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes attn_fwd_simple needs for these sizes (n_seq: the number of
 * sequences cu_seqlens will describe, 1 without cu_seqlens); host-only.  Large
 * enough for any key-split count the library may choose on the current device;
 * 0 for n_seq < 1. */
ATTN_API size_t attn_fwd_simple_workspace_bytes(int32_t N, int32_t H, int32_t D, int32_t relation,
                                                int32_t n_seq, int32_t dtype);

/* The kernel family a call with these arguments runs (ATTN_KERNEL_SIMT or
 * ATTN_KERNEL_TC, resolving AUTO), or a negative attn_status if the call
 * would be rejected.  Host-only; launches nothing. */
ATTN_API int attn_fwd_selected_kernel(const attn_fwd_args *a);
ATTN_API int attn_bwd_selected_kernel(const attn_bwd_args *a);

/* The dq mode a backward with these arguments runs (ATTN_DQ_SEPARATE or
 * ATTN_DQ_FUSED, resolving AUTO), or a negative attn_status.  Host-only. */
ATTN_API int attn_bwd_selected_dq_mode(const attn_bwd_args *a);

/* Attention over the CSR relation of `a` (see attn_csr_args). */
ATTN_API int attn_csr_fwd(const attn_csr_args *a, void *stream);

/* Forward for callers that cannot allocate device memory (no counterpart on
 * the pages; a deployment convenience).  Same arguments and results as
 * attn_fwd, except that `num_splits` is taken as 1 (no key splits) and
 * `workspace` / `workspace_bytes` are ignored: the
 * scheduler's scratch lives in a fixed 64 KiB array inside this library's
 * device memory, which every GPU that loads the library keeps until the
 * process exits.  No call allocates anything.
 *  - n_seq must be at most ATTN_NOALLOC_MAX_SEQ; larger inputs return
 *    ATTN_EUNSUPPORTED before any launch.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    The address is kept per device ordinal, so calls must run in the
 *    device's primary context (the CUDA runtime's default context).
 *  - All calls share the one array and each call rewrites the part it reads,
 *    so calls whose kernels overlap on the GPU (concurrent streams, or
 *    threads on one device) race: serialise them on one stream. */
#define ATTN_NOALLOC_MAX_SEQ 16367
ATTN_API int attn_fwd_noalloc(const attn_fwd_args *a, void *stream);

/* Bounded-wait budget, in SM clock cycles, of every mbarrier wait in the
 * tensor-core kernels launched after this call (default 4e9, or the
 * ATTN_WATCHDOG_CYCLES environment variable; cycles <= 0 restores that).  When
 * a wait runs out the kernel stops, drains its loads in flight, frees its
 * tensor memory and exits; attn_device_status() then returns ATTN_ETIMEOUT.
 * Budgets below 2^20 cycles (meant for failure-detection tests) make every
 * wait poll without suspending, so that they run out reliably; larger ones let
 * a wait suspend in hardware first.  Returns the previous budget. */
ATTN_API long long attn_set_watchdog_cycles(long long cycles);

/* Synchronises `stream`, then returns and clears the device-side status word
 * of the current device: ATTN_OK, ATTN_EINVAL (a kernel found inconsistent
 * cu_seqlens and skipped the work) or ATTN_ETIMEOUT (a bounded wait expired
 * and the kernel exited early; outputs are then incomplete). */
ATTN_API int attn_device_status(void *stream);

/* Diagnostic: y[i] = 2^x[i] computed by the polynomial exp2 that the
 * tensor-core kernels run on the FMA pipe for part of the softmax (Cody-Waite
 * range reduction, degree-4 polynomial; max relative error 2.9e-6 for
 * -126 <= x <= 127; x is clamped to that range first, so larger arguments
 * give about 2^127 and smaller ones about 2^-126).  x, y: device arrays of n
 * floats. */
ATTN_API int attn_selftest_exp2(const float *x, float *y, int32_t n, void *stream);

/* Number of kernels the library has launched in this process (all devices). */
ATTN_API uint64_t attn_launch_count(void);

/* Static text for a status code, and the last CUDA error text of this thread. */
ATTN_API const char *attn_strerror(int code);
ATTN_API const char *attn_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */

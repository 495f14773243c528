// C ABI of the attention library: argument validation, workspace layout,
// schedule preparation and kernel dispatch.  See include/attn.h for the
// contract of each entry point.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/attn.h"
#include "internal.h"
#include "tc.h"

namespace attn {

namespace {

__device__ int g_status;  // first error reported by a kernel on this device

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::atomic<uint64_t> g_launches{0};
thread_local std::string g_last_error;

int set_cuda_error(cudaError_t e) {
    g_last_error = cudaGetErrorString(e);
    return ATTN_ECUDA;
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int *status_ptr() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

constexpr long long kDefaultWatchdog = 4000000000LL;  // about 2 s at 2 GHz per bounded wait
std::atomic<long long> g_watchdog{0};

long long watchdog_cycles() {
    long long v = g_watchdog.load(std::memory_order_relaxed);
    if (v > 0) return v;
    const char *e = std::getenv("ATTN_WATCHDOG_CYCLES");
    const long long x = e ? std::atoll(e) : 0;
    return x > 0 ? x : kDefaultWatchdog;
}

// ATTN_LOG=1 in the environment: one line on stderr per forward / backward
// call naming the schedule the library chose (kernel family, key splits, dq
// mode).  Off by default.
bool log_on() {
    static const bool on = [] {
        const char *e = std::getenv("ATTN_LOG");
        return e && std::atoi(e) > 0;
    }();
    return on;
}

const char *dtype_name(int dt) { return dt == ATTN_F16 ? "f16" : dt == ATTN_BF16 ? "bf16" : "f32"; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t elem_size(int dt) { return dt == ATTN_F32 ? 4 : 2; }

bool valid_dtype(int dt) { return dt == ATTN_F16 || dt == ATTN_BF16 || dt == ATTN_F32; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// A tensor view is usable when its pointer and row strides keep every
// D-element row 16-byte aligned.
bool valid_view_bytes(const attn_tensor &t, int64_t es, bool required) {
    if (!t.ptr) return !required;
    if (!aligned16(t.ptr)) return false;
    if (t.stride_tok <= 0 || t.stride_head <= 0) return false;
    return (t.stride_tok * es) % 16 == 0 && (t.stride_head * es) % 16 == 0;
}

bool valid_view(const attn_tensor &t, int dt, bool required) {
    return valid_view_bytes(t, (int64_t)elem_size(dt), required);
}

// Which implementation runs: true = tcgen05 kernels.  `tc_ok` says whether
// the tensor-core kernels cover the arguments.
int choose_tc(int kernel, bool tc_ok, bool &use_tc) {
    if (kernel == ATTN_KERNEL_SIMT) {
        use_tc = false;
        return ATTN_OK;
    }
    if (kernel == ATTN_KERNEL_TC) {
        if (!tc_ok) return ATTN_EUNSUPPORTED;
        use_tc = true;
        return ATTN_OK;
    }
    if (kernel != ATTN_KERNEL_AUTO) return ATTN_EINVAL;
    use_tc = tc_ok;
    return ATTN_OK;
}

int check_common(int n_q, int n_k, int H, int D, int relation, int dtype, int n_seq,
                 const int32_t *cu_q, const int32_t *cu_k, float scale) {
    if (n_q < 0 || n_k < 0 || H < 1 || n_seq < 1) return ATTN_EINVAL;
    if (!valid_dtype(dtype)) return ATTN_EINVAL;
    if (relation != ATTN_FULL && relation != ATTN_CAUSAL) return ATTN_EINVAL;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return ATTN_EINVAL;
    if ((cu_q == nullptr) != (cu_k == nullptr)) return ATTN_EINVAL;
    if (!cu_q && n_seq != 1) return ATTN_EINVAL;
    if (!cu_q && relation == ATTN_CAUSAL && n_q != n_k) return ATTN_EUNSUPPORTED;
    if (D != 64 && D != 128) return ATTN_EUNSUPPORTED;
    // work-item numbering is int32: H * (tiles + sequences) must fit
    const int64_t items = (int64_t)H * ((int64_t)(n_q > n_k ? n_q : n_k) / kSimtBlock + n_seq + 1);
    if (items >= (int64_t)1 << 31 || (int64_t)n_q * H >= (int64_t)1 << 31) return ATTN_EUNSUPPORTED;
    return ATTN_OK;
}

size_t sched_bytes(int n_seq) { return align256(sizeof(int) * (size_t)(kSchedHeaderInts + n_seq + 1)); }

Sched sched_at(void *base) {
    int *p = static_cast<int *>(base);
    return Sched{p, p + kSchedHeaderInts};
}

// ---- forward ---------------------------------------------------------------

// Split-K choice when the caller leaves it to the library: split only when the
// query tiles alone fill less than half of the resident CTA slots, into as
// many chunks as fill the slots once, keeping at least two key tiles per chunk
// (of the average sequence; the causal relation halves the keys a tile scans
// on average).
int auto_splits(const FwdParams &p, bool use_tc) {
    const int64_t q_block = use_tc ? tc_fwd_block_rows(p) : kSimtBlock;
    const int64_t k_block = use_tc ? 128 : 64;
    const int64_t per_seq_q = p.n_q / p.n_seq, per_seq_k = p.n_k / p.n_seq;
    const int64_t q_tiles = (int64_t)p.n_seq * ((per_seq_q + q_block - 1) / q_block);
    const int64_t items = (q_tiles > 0 ? q_tiles : 1) * p.H;
    const int64_t slots = (int64_t)sm_count() * (use_tc ? 1 : fwd_simt_ctas_per_sm(p));
    if (2 * items > slots) return 1;
    int64_t k_tiles = (per_seq_k + k_block - 1) / k_block;
    if (p.causal) k_tiles /= 2;
    int64_t c = slots / items;
    if (c > k_tiles / 2) c = k_tiles / 2;
    if (c > ATTN_MAX_SPLITS) c = ATTN_MAX_SPLITS;
    return c >= 2 ? (int)c : 1;
}

struct FwdLayout {
    size_t o_parts, lse_parts, split_ops, total;
};

// Workspace of a forward: the schedule block; with key splits the f32 partial
// outputs and lse; for f32 inputs on the tensor cores the bf16 parts of q, k, v.
FwdLayout fwd_layout(int n_seq, int n_q, int H, int D, int splits, size_t op_bytes) {
    FwdLayout L;
    L.o_parts = sched_bytes(n_seq);
    L.lse_parts = L.o_parts;
    L.split_ops = L.o_parts;
    if (splits > 1) {
        const size_t rows = (size_t)splits * (size_t)n_q * (size_t)H;
        L.lse_parts = L.o_parts + align256(sizeof(float) * rows * (size_t)D);
        L.split_ops = L.lse_parts + align256(sizeof(float) * rows);
    }
    L.total = L.split_ops + align256(op_bytes);
    return L;
}

// Bytes of the bf16 operand parts a forward with these parameters keeps in the
// workspace (f32 inputs on the tensor cores only).
size_t split_op_bytes(const FwdParams &p, bool use_tc) {
    return use_tc && p.dtype == ATTN_F32 ? x3_split_bytes(p.n_q, p.n_k, p.H) : 0;
}

FwdLayout fwd_layout_of(const FwdParams &p, bool use_tc) {
    return fwd_layout(p.n_seq, p.n_q, p.H, p.D, p.n_splits, split_op_bytes(p, use_tc));
}

// Validates everything but the workspace and fills the kernel parameters that
// do not depend on it; resolves the kernel family and the key splits.  With
// `check_views` false the tensor pointers and strides are not looked at (the
// workspace size depends on sizes only, so a caller may size it before its
// tensors exist).
int plan_fwd(const attn_fwd_args *a, FwdParams &p, bool &use_tc, bool check_views = true) {
    if (!a) return ATTN_EINVAL;
    int rc = check_common(a->n_q, a->n_k, a->H, a->D, a->relation, a->dtype, a->n_seq,
                          a->cu_seqlens_q, a->cu_seqlens_k, a->scale);
    if (rc) return rc;
    if (a->o_dtype != a->dtype && a->o_dtype != ATTN_F32) return ATTN_EINVAL;
    if (a->num_splits < 0 || a->num_splits > ATTN_MAX_SPLITS) return ATTN_EINVAL;
    const float rho = a->prune_threshold;
    if (!(rho >= 0.f && rho <= 1.f)) return ATTN_EINVAL;  // also rejects NaN
    // tile pruning is defined for the dense relation over one sequence, unsplit
    if (rho > 0.f && (a->relation != ATTN_FULL || a->cu_seqlens_q || a->num_splits > 1))
        return ATTN_EUNSUPPORTED;
    if (a->qk_fp8 != 0 && a->qk_fp8 != 1) return ATTN_EINVAL;
    // fp8 Q / K: tensor-core kernels, V (and P) 16-bit, D = 128, positive scale
    if (a->qk_fp8 && (a->dtype == ATTN_F32 || a->D != 128 || !(a->scale > 0.f) ||
                      a->kernel == ATTN_KERNEL_SIMT))
        return ATTN_EUNSUPPORTED;
    const bool any_q = a->n_q > 0, any_k = a->n_k > 0;
    const bool qk_ok = a->qk_fp8 ? valid_view_bytes(a->q, 1, any_q) && valid_view_bytes(a->k, 1, any_k)
                                 : valid_view(a->q, a->dtype, any_q) && valid_view(a->k, a->dtype, any_k);
    if (check_views &&
        (!qk_ok || !valid_view(a->o, a->o_dtype, any_q) || !valid_view(a->v, a->dtype, any_k)))
        return ATTN_EINVAL;
    std::memset(&p, 0, sizeof(p));
    p.qk_fp8 = a->qk_fp8;
    p.q = a->q.ptr; p.k = a->k.ptr; p.v = a->v.ptr; p.o = a->o.ptr; p.lse = a->lse;
    p.q_st = a->q.stride_tok; p.q_sh = a->q.stride_head;
    p.k_st = a->k.stride_tok; p.k_sh = a->k.stride_head;
    p.v_st = a->v.stride_tok; p.v_sh = a->v.stride_head;
    p.o_st = a->o.stride_tok; p.o_sh = a->o.stride_head;
    p.n_q = a->n_q; p.n_k = a->n_k; p.H = a->H; p.D = a->D;
    p.scale = a->scale;
    p.scale_log2 = a->scale * 1.4426950408889634f;
    p.causal = a->relation == ATTN_CAUSAL;
    p.dtype = a->dtype; p.o_dtype = a->o_dtype;
    p.n_seq = a->n_seq;
    p.cu_q = a->cu_seqlens_q; p.cu_k = a->cu_seqlens_k;
    p.watchdog_cycles = watchdog_cycles();
    p.prune = rho > 0.f;
    p.prune_log2 = p.prune ? std::log2(rho) : 0.f;
    p.pruned_tiles = reinterpret_cast<unsigned long long *>(a->pruned_tiles);
    rc = choose_tc(a->kernel, tc_fwd_supported(p), use_tc);
    if (rc) return rc;
    if (p.qk_fp8 && !use_tc) return ATTN_EUNSUPPORTED;  // no CUDA-core fp8 path
    p.n_splits = p.prune ? 1 : (a->num_splits > 0 ? a->num_splits : auto_splits(p, use_tc));
    // work items (tiles x heads x splits) are numbered in int32
    const int64_t tiles = (int64_t)a->H * ((int64_t)a->n_q / kSimtBlock + a->n_seq + 1);
    if (tiles * p.n_splits >= (int64_t)1 << 31) return ATTN_EUNSUPPORTED;
    return ATTN_OK;
}

int build_fwd(const attn_fwd_args *a, FwdParams &p, bool &use_tc) {
    int rc = plan_fwd(a, p, use_tc);
    if (rc) return rc;
    const FwdLayout L = fwd_layout_of(p, use_tc);
    if (!a->workspace || a->workspace_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(a->workspace) & 255))
        return ATTN_EWORKSPACE;
    p.sched = sched_at(a->workspace);
    p.split_ws = split_op_bytes(p, use_tc) ? static_cast<char *>(a->workspace) + L.split_ops : nullptr;
    p.status = status_ptr();
    if (!p.status) return ATTN_ECUDA;
    return ATTN_OK;
}

// Kernel parameters of the split-K partial pass and of its merge: the
// attention kernel writes chunk c's O_c (f32, token stride H*D, head stride D)
// and lse_c into the workspace; the merge writes the caller's o and lse.
void split_params(const attn_fwd_args *a, const FwdParams &p, bool use_tc, FwdParams &part, MergeParams &m) {
    const FwdLayout L = fwd_layout_of(p, use_tc);
    char *ws = static_cast<char *>(a->workspace);
    float *o_parts = reinterpret_cast<float *>(ws + L.o_parts);
    float *lse_parts = reinterpret_cast<float *>(ws + L.lse_parts);
    part = p;
    part.o = o_parts;
    part.o_dtype = ATTN_F32;
    part.o_st = (int64_t)a->H * a->D;
    part.o_sh = a->D;
    part.o_split_st = (int64_t)a->n_q * a->H * a->D;
    part.lse = lse_parts;
    part.lse_split_st = (int64_t)a->H * a->n_q;
    std::memset(&m, 0, sizeof(m));
    m.o_parts = o_parts;
    m.lse_parts = lse_parts;
    m.o = a->o.ptr;
    m.lse = a->lse;
    m.o_st = a->o.stride_tok;
    m.o_sh = a->o.stride_head;
    m.part_st = part.o_split_st;
    m.n_parts = p.n_splits;
    m.n_q = a->n_q;
    m.H = a->H;
    m.D = a->D;
    m.o_dtype = a->o_dtype;
}

// ---- backward --------------------------------------------------------------

struct BwdLayout {
    size_t kv, q, dr, lse2, dqa, total;
};

// fused: room for the dq partial sums (n_q * H * D f32) after the row statistics
BwdLayout bwd_layout(int n_seq, int H, int n_q, int D, bool fused) {
    BwdLayout L;
    const size_t rows = align256(sizeof(float) * (size_t)H * (size_t)(n_q > 0 ? n_q : 1));
    L.kv = 0;
    L.q = sched_bytes(n_seq);
    L.dr = L.q + sched_bytes(n_seq);
    L.lse2 = L.dr + rows;
    L.dqa = L.lse2 + rows;
    L.total = L.dqa + (fused ? align256(sizeof(float) * (size_t)H * (size_t)(n_q > 0 ? n_q : 0) * (size_t)D) : 0);
    return L;
}

// Whether a backward with these arguments accumulates dq inside the dK/dV
// kernel: the caller asked for it and the tensor-core kernels run (AUTO
// resolves to the separate dq kernel).
bool bwd_fused(const attn_bwd_args *a) {
    if (a->dq_mode != ATTN_DQ_FUSED) return false;
    BwdParams t;
    std::memset(&t, 0, sizeof(t));
    t.dtype = a->dtype;
    t.D = a->D;
    t.n_q = a->n_q;
    t.n_k = a->n_k;
    bool use_tc = false;
    if (choose_tc(a->kernel, tc_bwd_supported(t), use_tc) != ATTN_OK) return false;
    return use_tc;
}

int build_bwd(const attn_bwd_args *a, BwdParams &p, bool &use_tc) {
    if (!a) return ATTN_EINVAL;
    int rc = check_common(a->n_q, a->n_k, a->H, a->D, a->relation, a->dtype, a->n_seq,
                          a->cu_seqlens_q, a->cu_seqlens_k, a->scale);
    if (rc) return rc;
    if (a->o_dtype != a->dtype && a->o_dtype != ATTN_F32) return ATTN_EINVAL;
    if (a->grad_dtype != a->dtype && a->grad_dtype != ATTN_F32) return ATTN_EINVAL;
    if (a->prune_threshold != 0.f) return ATTN_EUNSUPPORTED;  // fails closed
    if (a->dq_mode != ATTN_DQ_AUTO && a->dq_mode != ATTN_DQ_SEPARATE && a->dq_mode != ATTN_DQ_FUSED)
        return ATTN_EINVAL;
    const bool any_q = a->n_q > 0, any_k = a->n_k > 0;
    if (!valid_view(a->q, a->dtype, any_q) || !valid_view(a->o, a->o_dtype, any_q) ||
        !valid_view(a->dout, a->dtype, any_q) || !valid_view(a->dq, a->grad_dtype, any_q) ||
        !valid_view(a->k, a->dtype, any_k) || !valid_view(a->v, a->dtype, any_k) ||
        !valid_view(a->dk, a->grad_dtype, any_k) || !valid_view(a->dv, a->grad_dtype, any_k))
        return ATTN_EINVAL;
    if (any_q && !a->lse) return ATTN_EINVAL;
    if (!a->workspace || a->workspace_bytes < attn_bwd_workspace_bytes(a) ||
        (reinterpret_cast<uintptr_t>(a->workspace) & 255))
        return ATTN_EWORKSPACE;
    std::memset(&p, 0, sizeof(p));
    p.q = a->q.ptr; p.k = a->k.ptr; p.v = a->v.ptr; p.o = a->o.ptr; p.dout = a->dout.ptr;
    p.lse = a->lse; p.dq = a->dq.ptr; p.dk = a->dk.ptr; p.dv = a->dv.ptr;
    p.q_st = a->q.stride_tok; p.q_sh = a->q.stride_head;
    p.k_st = a->k.stride_tok; p.k_sh = a->k.stride_head;
    p.v_st = a->v.stride_tok; p.v_sh = a->v.stride_head;
    p.o_st = a->o.stride_tok; p.o_sh = a->o.stride_head;
    p.do_st = a->dout.stride_tok; p.do_sh = a->dout.stride_head;
    p.dq_st = a->dq.stride_tok; p.dq_sh = a->dq.stride_head;
    p.dk_st = a->dk.stride_tok; p.dk_sh = a->dk.stride_head;
    p.dv_st = a->dv.stride_tok; p.dv_sh = a->dv.stride_head;
    p.n_q = a->n_q; p.n_k = a->n_k; p.H = a->H; p.D = a->D;
    p.scale = a->scale;
    p.scale_log2 = a->scale * 1.4426950408889634f;
    p.causal = a->relation == ATTN_CAUSAL;
    p.dtype = a->dtype; p.o_dtype = a->o_dtype; p.grad_dtype = a->grad_dtype;
    p.n_seq = a->n_seq;
    p.cu_q = a->cu_seqlens_q; p.cu_k = a->cu_seqlens_k;
    const bool fused = bwd_fused(a);
    const BwdLayout L = bwd_layout(a->n_seq, a->H, a->n_q, a->D, fused);
    char *ws = static_cast<char *>(a->workspace);
    p.sched_kv = sched_at(ws + L.kv);
    p.sched_q = sched_at(ws + L.q);
    p.dr = reinterpret_cast<float *>(ws + L.dr);
    p.lse2 = reinterpret_cast<float *>(ws + L.lse2);
    p.dq_accum = fused ? reinterpret_cast<float *>(ws + L.dqa) : nullptr;
    p.status = status_ptr();
    p.watchdog_cycles = watchdog_cycles();
    if (!p.status) return ATTN_ECUDA;
    rc = choose_tc(a->kernel, tc_bwd_supported(p), use_tc);
    if (rc) return rc;
    if (a->dq_mode == ATTN_DQ_FUSED && !use_tc) return ATTN_EUNSUPPORTED;
    return ATTN_OK;
}

}  // namespace

int sm_count() {
    const int dev = current_device();
    if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev] = n;
    return n;
}

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace attn

using namespace attn;

extern "C" {

int attn_abi_version(void) { return ATTN_ABI_VERSION; }
size_t attn_fwd_args_size(void) { return sizeof(attn_fwd_args); }
size_t attn_bwd_args_size(void) { return sizeof(attn_bwd_args); }
uint64_t attn_launch_count(void) { return g_launches.load(); }

size_t attn_fwd_workspace_bytes(const attn_fwd_args *a) {
    if (!a || a->n_seq < 1) return 0;
    FwdParams p;
    bool use_tc = false;
    // arguments the forward would reject need no split buffers
    if (plan_fwd(a, p, use_tc, false) == ATTN_OK) return fwd_layout_of(p, use_tc).total;
    return fwd_layout(a->n_seq, a->n_q > 0 ? a->n_q : 0, a->H > 0 ? a->H : 0, a->D > 0 ? a->D : 0, 1, 0)
        .total;
}

size_t attn_merge_args_size(void) { return sizeof(attn_merge_args); }

size_t attn_bwd_workspace_bytes(const attn_bwd_args *a) {
    if (!a || a->n_seq < 1 || a->H < 1 || a->n_q < 0 || a->D < 0) return 0;
    return bwd_layout(a->n_seq, a->H, a->n_q, a->D, bwd_fused(a)).total;
}

int attn_fwd(const attn_fwd_args *a, void *stream) {
    FwdParams p;
    bool use_tc = false;
    int rc = build_fwd(a, p, use_tc);
    if (rc) return rc;
    if (a->n_q == 0) return ATTN_OK;
    if (log_on())
        std::fprintf(stderr,
                     "[attn] fwd n_q=%d n_k=%d H=%d D=%d n_seq=%d relation=%s dtype=%s%s o_dtype=%s "
                     "kernel=%s splits=%d prune=%g\n",
                     a->n_q, a->n_k, a->H, a->D, a->n_seq, p.causal ? "causal" : "full",
                     p.qk_fp8 ? "e4m3+" : "", dtype_name(a->dtype), dtype_name(a->o_dtype),
                     use_tc ? "tc" : "simt", p.n_splits, (double)a->prune_threshold);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int block = use_tc ? tc_fwd_block_rows(p) : kSimtBlock;
    // One sequence whose work items all fit in one wave of the default grid:
    // static schedule (CTA i runs item i), no preparation launch.
    const int64_t items = ((int64_t)p.n_q + block - 1) / block * p.H * p.n_splits;
    if (!p.cu_q && a->num_ctas == 0 &&
        items <= (int64_t)sm_count() * (use_tc ? 1 : fwd_simt_ctas_per_sm(p)))
        p.static_items = (int)items;
    cudaError_t e = cudaSuccess;
    if (!p.static_items)
        e = launch_prep(p.cu_q, p.cu_k, p.n_seq, p.n_q, p.n_k, p.H, block, p.causal, 0, p.n_splits,
                        p.sched, p.status, s);
    if (e != cudaSuccess) return set_cuda_error(e);
    const int grid = p.static_items ? p.static_items : a->num_ctas;
    if (p.n_splits == 1) {
        e = use_tc ? launch_fwd_tc(p, grid, s) : launch_fwd_simt(p, grid, s);
    } else {
        FwdParams part;
        MergeParams m;
        split_params(a, p, use_tc, part, m);
        e = use_tc ? launch_fwd_tc(part, grid, s) : launch_fwd_simt(part, grid, s);
        if (e == cudaSuccess) e = launch_merge(m, s);
    }
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

int attn_fwd_num_splits(const attn_fwd_args *a) {
    FwdParams p;
    bool use_tc = false;
    const int rc = plan_fwd(a, p, use_tc);
    return rc ? rc : p.n_splits;
}

int attn_merge(const attn_merge_args *a, void *stream) {
    if (!a) return ATTN_EINVAL;
    if (a->n_parts < 1 || a->n_parts > ATTN_MAX_SPLITS || a->n_q < 0 || a->H < 1 || a->D < 4 ||
        a->D > 256 || (a->D & 3) || !valid_dtype(a->o_dtype))
        return ATTN_EINVAL;
    if ((int64_t)a->n_q * a->H * a->n_parts >= (int64_t)1 << 31) return ATTN_EUNSUPPORTED;
    if (a->n_q == 0) return ATTN_OK;
    if (!a->o_parts || !aligned16(a->o_parts) || !a->lse_parts ||
        (reinterpret_cast<uintptr_t>(a->lse_parts) & 3) || !valid_view(a->o, a->o_dtype, true))
        return ATTN_EINVAL;
    MergeParams m;
    std::memset(&m, 0, sizeof(m));
    m.o_parts = a->o_parts;
    m.lse_parts = a->lse_parts;
    m.o = a->o.ptr;
    m.lse = a->lse;
    m.o_st = a->o.stride_tok;
    m.o_sh = a->o.stride_head;
    m.part_st = (int64_t)a->n_q * a->H * a->D;
    m.n_parts = a->n_parts;
    m.n_q = a->n_q;
    m.H = a->H;
    m.D = a->D;
    m.o_dtype = a->o_dtype;
    cudaError_t e = launch_merge(m, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

int attn_bwd_preprocess(const attn_bwd_args *a, void *stream) {
    BwdParams p;
    bool use_tc = false;
    int rc = build_bwd(a, p, use_tc);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kv_block = use_tc ? tc_bwd_kv_block(p) : kSimtBlock;
    const int q_block = use_tc ? tc_bwd_q_block(p) : kSimtBlock;
    cudaError_t e = launch_prep(p.cu_q, p.cu_k, p.n_seq, p.n_q, p.n_k, p.H, kv_block, p.causal, 1,
                                1, p.sched_kv, p.status, s);
    if (e == cudaSuccess && !p.dq_accum)  // the fused dq needs no query-block schedule
        e = launch_prep(p.cu_q, p.cu_k, p.n_seq, p.n_q, p.n_k, p.H, q_block, p.causal, 0,
                        1, p.sched_q, p.status, s);
    if (e == cudaSuccess) e = launch_bwd_preprocess(p, s);
    if (e == cudaSuccess && p.dq_accum) e = launch_dq_accum_zero(p, s);
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

int attn_bwd_dkdv(const attn_bwd_args *a, void *stream) {
    BwdParams p;
    bool use_tc = false;
    int rc = build_bwd(a, p, use_tc);
    if (rc) return rc;
    if (a->n_k == 0) return ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = use_tc ? launch_bwd_dkdv_tc(p, a->num_ctas, s)
                           : launch_bwd_dkdv_simt(p, a->num_ctas, s);
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

int attn_bwd_dq(const attn_bwd_args *a, void *stream) {
    BwdParams p;
    bool use_tc = false;
    int rc = build_bwd(a, p, use_tc);
    if (rc) return rc;
    if (a->n_q == 0) return ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = p.dq_accum ? launch_dq_accum_convert(p, s)
                    : use_tc   ? launch_bwd_dq_tc(p, a->num_ctas, s)
                               : launch_bwd_dq_simt(p, a->num_ctas, s);
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

int attn_bwd(const attn_bwd_args *a, void *stream) {
    if (log_on()) {
        BwdParams p;
        bool use_tc = false;
        if (build_bwd(a, p, use_tc) == ATTN_OK)
            std::fprintf(stderr,
                         "[attn] bwd n_q=%d n_k=%d H=%d D=%d n_seq=%d relation=%s dtype=%s "
                         "grad_dtype=%s kernel=%s dq=%s\n",
                         a->n_q, a->n_k, a->H, a->D, a->n_seq, p.causal ? "causal" : "full",
                         dtype_name(a->dtype), dtype_name(a->grad_dtype), use_tc ? "tc" : "simt",
                         p.dq_accum ? "fused" : "separate");
    }
    int rc = attn_bwd_preprocess(a, stream);
    if (rc) return rc;
    rc = attn_bwd_dkdv(a, stream);
    if (rc) return rc;
    return attn_bwd_dq(a, stream);
}

}  // extern "C"

namespace {

// The argument struct of the flat form: contiguous (N, H, D) tensors (token
// stride H * D, head stride D), o in the input dtype, AUTO kernel and splits.
attn_fwd_args simple_args(const void *q, const void *k, const void *v, void *out, float *lse,
                          int32_t N, int32_t H, int32_t D, float scale, int32_t relation,
                          const int32_t *cu_seqlens, int32_t n_seq, int32_t dtype) {
    attn_fwd_args a;
    std::memset(&a, 0, sizeof(a));
    const int64_t st = (int64_t)H * D;
    a.q = attn_tensor{const_cast<void *>(q), st, D};
    a.k = attn_tensor{const_cast<void *>(k), st, D};
    a.v = attn_tensor{const_cast<void *>(v), st, D};
    a.o = attn_tensor{out, st, D};
    a.lse = lse;
    a.n_q = a.n_k = N;
    a.H = H;
    a.D = D;
    a.scale = scale;
    a.relation = relation;
    a.dtype = a.o_dtype = dtype;
    a.n_seq = cu_seqlens ? n_seq : 1;
    a.cu_seqlens_q = a.cu_seqlens_k = cu_seqlens;
    a.kernel = ATTN_KERNEL_AUTO;
    return a;
}

}  // namespace

extern "C" {

int attn_fwd_simple(const void *q, const void *k, const void *v, void *out, float *lse,
                    int32_t N, int32_t H, int32_t D, float scale, int32_t relation,
                    const int32_t *cu_seqlens, int32_t n_seq, int32_t dtype, void *workspace,
                    size_t workspace_bytes, void *stream) {
    attn_fwd_args a = simple_args(q, k, v, out, lse, N, H, D, scale, relation, cu_seqlens, n_seq, dtype);
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return attn_fwd(&a, stream);
}

size_t attn_fwd_simple_workspace_bytes(int32_t N, int32_t H, int32_t D, int32_t relation,
                                       int32_t n_seq, int32_t dtype) {
    if (n_seq < 1) return 0;
    // only the presence of cu_seqlens matters for the size (n_seq > 1 needs it);
    // this placeholder is never dereferenced
    static const int32_t placeholder[2] = {0, 0};
    const attn_fwd_args a = simple_args(nullptr, nullptr, nullptr, nullptr, nullptr, N, H, D, 1.f,
                                        relation, n_seq > 1 ? placeholder : nullptr, n_seq, dtype);
    return attn_fwd_workspace_bytes(&a);
}

int attn_fwd_selected_kernel(const attn_fwd_args *a) {
    FwdParams p;
    bool use_tc = false;
    const int rc = build_fwd(a, p, use_tc);
    return rc ? rc : (use_tc ? ATTN_KERNEL_TC : ATTN_KERNEL_SIMT);
}

int attn_bwd_selected_kernel(const attn_bwd_args *a) {
    BwdParams p;
    bool use_tc = false;
    const int rc = build_bwd(a, p, use_tc);
    return rc ? rc : (use_tc ? ATTN_KERNEL_TC : ATTN_KERNEL_SIMT);
}

int attn_bwd_selected_dq_mode(const attn_bwd_args *a) {
    BwdParams p;
    bool use_tc = false;
    const int rc = build_bwd(a, p, use_tc);
    return rc ? rc : (p.dq_accum ? ATTN_DQ_FUSED : ATTN_DQ_SEPARATE);
}

long long attn_set_watchdog_cycles(long long cycles) {
    const long long prev = watchdog_cycles();
    g_watchdog.store(cycles > 0 ? cycles : 0, std::memory_order_relaxed);
    return prev;
}

int attn_device_status(void *stream) {
    int *sp = status_ptr();
    if (!sp) return ATTN_ECUDA;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return set_cuda_error(e);
    int v = 0;
    e = cudaMemcpy(&v, sp, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(sp, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return set_cuda_error(e);
    }
    return v;
}

size_t attn_csr_args_size(void) { return sizeof(attn_csr_args); }

int attn_csr_fwd(const attn_csr_args *a, void *stream) {
    if (!a) return ATTN_EINVAL;
    if (a->n_dst < 0 || a->n_src < 0 || a->n_edges < 0 || a->H < 1 || a->D < 4 || a->D > 256 ||
        (a->D & 3) || !valid_dtype(a->dtype) || (a->o_dtype != a->dtype && a->o_dtype != ATTN_F32))
        return ATTN_EINVAL;
    const bool dot = a->edge_scores == nullptr;
    if (dot && !(a->scale == a->scale && a->scale != INFINITY && a->scale != -INFINITY))
        return ATTN_EINVAL;
    if ((int64_t)a->n_dst * a->H >= ((int64_t)1 << 40)) return ATTN_EUNSUPPORTED;
    if (a->n_dst == 0) return ATTN_OK;
    const bool any_e = a->n_edges > 0;
    if (!a->row_ptr || (any_e && !a->col_idx) || (reinterpret_cast<uintptr_t>(a->row_ptr) & 7) ||
        (reinterpret_cast<uintptr_t>(a->col_idx) & 3) ||
        (!dot && (reinterpret_cast<uintptr_t>(a->edge_scores) & 3)) ||
        (reinterpret_cast<uintptr_t>(a->row_order) & 3))
        return ATTN_EINVAL;
    if (!valid_view(a->o, a->o_dtype, true) || !valid_view(a->v, a->dtype, any_e && a->n_src > 0) ||
        (dot && (!valid_view(a->q, a->dtype, true) || !valid_view(a->k, a->dtype, any_e && a->n_src > 0))))
        return ATTN_EINVAL;
    CsrParams p;
    std::memset(&p, 0, sizeof(p));
    p.row_ptr = a->row_ptr;
    p.col = a->col_idx;
    p.n_edges = a->n_edges;
    p.n_dst = a->n_dst;
    p.n_src = a->n_src;
    p.H = a->H;
    p.D = a->D;
    p.scores = a->edge_scores;
    p.q = a->q.ptr; p.k = a->k.ptr; p.v = a->v.ptr; p.o = a->o.ptr; p.lse = a->lse;
    p.q_st = a->q.stride_tok; p.q_sh = a->q.stride_head;
    p.k_st = a->k.stride_tok; p.k_sh = a->k.stride_head;
    p.v_st = a->v.stride_tok; p.v_sh = a->v.stride_head;
    p.o_st = a->o.stride_tok; p.o_sh = a->o.stride_head;
    p.scale_log2 = a->scale * 1.4426950408889634f;
    p.dtype = a->dtype;
    p.o_dtype = a->o_dtype;
    p.row_order = a->row_order;
    p.status = status_ptr();
    if (!p.status) return ATTN_ECUDA;
    cudaError_t e = launch_csr_fwd(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return set_cuda_error(e);
    return ATTN_OK;
}

const char *attn_strerror(int code) {
    switch (code) {
    case ATTN_OK: return "success";
    case ATTN_EINVAL: return "invalid argument";
    case ATTN_EUNSUPPORTED: return "unsupported argument combination";
    case ATTN_ECUDA: return "CUDA runtime error";
    case ATTN_ETIMEOUT: return "device watchdog timeout";
    case ATTN_EWORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
    }
}

const char *attn_last_error_string(void) { return g_last_error.c_str(); }

}  // extern "C"

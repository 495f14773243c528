// attn_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers hold only their input and output buffers: a plugin or custom
// operator invoked by a host framework that owns every device allocation and
// hands out no allocator or workspace, or a steady-state serving loop that
// must not call cudaMalloc (it can synchronise the device and fragment a
// pre-sized memory pool).  For them this entry point takes the forward's
// scratch (the scheduler's work counter and per-sequence prefix) from a
// fixed-size array in this library's own device memory instead of a caller
// workspace.  Everything else -- validation, kernels, results -- is the
// regular attn_fwd.
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/attn.h"

namespace {

// Fixed scratch: every GPU that loads the library holds these 64 KiB until the
// process exits.  It fits the schedule of up to ATTN_NOALLOC_MAX_SEQ sequences.
constexpr size_t kScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_dev[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_dev[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_dev[dev] = p;
    }
    return g_scratch_dev[dev];
}

}  // namespace

extern "C" int attn_fwd_noalloc(const attn_fwd_args *a, void *stream) {
    if (!a) return ATTN_EINVAL;
    if (a->n_seq < 1) return ATTN_EINVAL;
    if (a->n_seq > ATTN_NOALLOC_MAX_SEQ) return ATTN_EUNSUPPORTED;  // beyond the fixed scratch
    attn_fwd_args b;
    std::memcpy(&b, a, sizeof(b));
    b.workspace = nullptr;
    b.workspace_bytes = 0;
    b.num_splits = 1;  // split-K partials would need more scratch than the fixed array
    // the tensor-core f32 forward keeps bf16 parts of q, k, v in its workspace:
    // f32 inputs take the CUDA-core kernel here unless the caller insists
    if (b.dtype == ATTN_F32 && b.kernel == ATTN_KERNEL_AUTO) b.kernel = ATTN_KERNEL_SIMT;
    if (attn_fwd_workspace_bytes(&b) > kScratchBytes) return ATTN_EUNSUPPORTED;
    void *scratch = scratch_address();
    if (!scratch) return ATTN_ECUDA;
    b.workspace = scratch;
    b.workspace_bytes = kScratchBytes;
    return attn_fwd(&b, stream);
}

// Host-side helpers of the tensor-core kernels: TMA tensor-map encoding
// (through the driver entry point, so the library does not link libcuda) and
// the device check.
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "tc.h"

namespace attn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

bool device_is_sm103() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3;
}

}  // namespace

bool tc_device_ok() {
    static const bool ok = device_is_sm103() && encode_fn() != nullptr;
    return ok;
}

bool make_tile_map(CUtensorMap *m, const void *ptr, int dtype, int D, int tokens, int H, int64_t st,
                   int64_t sh, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    const bool f8 = dtype == kDtypeE4M3;
    const cuuint64_t es_bytes = f8 ? 1 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)tokens, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)st * es_bytes, (cuuint64_t)sh * es_bytes};
    cuuint32_t box[3] = {f8 ? 128u : 64u, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn

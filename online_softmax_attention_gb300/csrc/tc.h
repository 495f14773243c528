// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once

#include <cuda.h>

#include "internal.h"

namespace attn {

// True on an sm_103 device with the driver's tensor-map encoder available.
bool tc_device_ok();

// Internal element-type code of fp8 (e4m3) Q / K tensors for make_tile_map.
constexpr int kDtypeE4M3 = 16;

// (tokens, heads, D) tensor -> 3-D TMA map {D, tokens, heads} with a box of
// `box_rows` rows x 128 bytes ({64, rows, 1} elements for 16-bit types,
// {128, rows, 1} for e4m3) and 128-byte swizzle.  False if the encoder rejects it.
bool make_tile_map(CUtensorMap *m, const void *ptr, int dtype, int D, int tokens, int H,
                   int64_t stride_tok, int64_t stride_head, int box_rows = 128);

// Whether the tensor-core kernels cover these arguments (dtype, D, strides).
bool tc_fwd_supported(const FwdParams &p);
bool tc_bwd_supported(const BwdParams &p);

// Rows of one forward / backward work item, for the schedule preparation.
int tc_fwd_block_rows(const FwdParams &p);
int tc_bwd_kv_block(const BwdParams &p);
int tc_bwd_q_block(const BwdParams &p);

cudaError_t launch_fwd_tc(const FwdParams &p, int num_ctas, cudaStream_t s);

// f32 inputs at D = 64 on the tensor cores (bf16 operand splitting, fwd_x3.cu):
// whether it covers the arguments, the workspace bytes of the operand parts,
// and the launch (the split prepass, then the attention kernel).
bool x3_fwd_supported(const FwdParams &p);
size_t x3_split_bytes(int n_q, int n_k, int H);
cudaError_t launch_fwd_x3(const FwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const BwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dq_tc(const BwdParams &p, int num_ctas, cudaStream_t s);

}  // namespace attn

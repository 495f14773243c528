// Tensor-core (tcgen05 / TMEM / TMA) attention kernels for sm_103a.
#pragma once

#include "internal.h"

namespace attn {

// Whether the tensor-core kernels cover these arguments (dtype, D, strides).
bool tc_fwd_supported(const FwdParams &p);
bool tc_bwd_supported(const BwdParams &p);

// Rows of one forward / backward work item, for the schedule preparation.
int tc_fwd_block_rows(const FwdParams &p);
int tc_bwd_kv_block(const BwdParams &p);
int tc_bwd_q_block(const BwdParams &p);

cudaError_t launch_fwd_tc(const FwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const BwdParams &p, int num_ctas, cudaStream_t s);
cudaError_t launch_bwd_dq_tc(const BwdParams &p, int num_ctas, cudaStream_t s);

}  // namespace attn

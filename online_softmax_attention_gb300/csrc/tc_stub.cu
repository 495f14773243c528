// Placeholder until the tcgen05 backward kernels land: reports "not covered".
#include "tc.h"

namespace attn {

bool tc_bwd_supported(const BwdParams &) { return false; }
int tc_bwd_kv_block(const BwdParams &) { return 128; }
int tc_bwd_q_block(const BwdParams &) { return 128; }
cudaError_t launch_bwd_dkdv_tc(const BwdParams &, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dq_tc(const BwdParams &, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace attn
